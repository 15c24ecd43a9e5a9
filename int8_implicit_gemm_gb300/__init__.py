"""Python binding of ``libi8conv.so`` (INT8 NCxHWx<32> Conv2d fprop on GB300).

A thin ctypes layer: argument marshalling only, every step of the
convolution runs in the library's CUDA kernels.  PyTorch supplies device
memory and streams.  The function names match the C entry points declared in
``include/i8conv.h``; ``Plan`` wraps the plan handle.

There is no fallback: if the library is missing this module raises at import
time, and without a GB300 the calls fail with ``I8ConvError``.
"""
from __future__ import annotations

import ctypes
import os

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "_lib", "libi8conv.so")

# status codes (include/i8conv.h)
I8C_OK = 0
I8C_ERR_INVALID_ARG = 1
I8C_ERR_UNSUPPORTED = 2
I8C_ERR_MISALIGNED = 3
I8C_ERR_OVERFLOW_RISK = 4
I8C_ERR_CUDA = 5
I8C_ERR_TIMEOUT = 6
I8C_ERR_NO_DEVICE = 7
I8C_DEBUG_SKIP_FIRST_ARRIVE = 1
I8C_DEBUG_TRACE = 2


class I8ConvError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {status_string(status)} ({status})")


class ConvShape(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in
                ("N", "C", "H", "W", "K", "R", "S", "pad_h", "pad_w",
                 "stride_h", "stride_w", "dil_h", "dil_w")]

    @classmethod
    def of(cls, shape) -> "ConvShape":
        if isinstance(shape, ConvShape):
            return shape
        if isinstance(shape, dict):
            return cls(*[int(shape[n]) for n, _ in cls._fields_])
        return cls(*[int(v) for v in shape])

    def astuple(self):
        return tuple(getattr(self, n) for n, _ in self._fields_)


class Epilogue(ctypes.Structure):
    """i8c_epilogue: per-output-channel scale and bias (device pointers) and ReLU."""
    _fields_ = [("alpha", ctypes.c_void_p), ("bias", ctypes.c_void_p), ("relu", ctypes.c_int32)]


class Options(ctypes.Structure):
    _fields_ = [("block_n", ctypes.c_int32), ("num_ctas", ctypes.c_int32),
                ("max_chunk_slices", ctypes.c_int32), ("wait_timeout_us", ctypes.c_int32),
                ("host_staging", ctypes.c_int32), ("debug_flags", ctypes.c_int32),
                ("timing_events", ctypes.c_int32), ("kernel_variant", ctypes.c_int32),
                ("halo_loads", ctypes.c_int32), ("tail_split", ctypes.c_int32), ("tile_shape", ctypes.c_int32),
                ("fused_filter", ctypes.c_int32), ("tile_px", ctypes.c_int32), ("filter_run", ctypes.c_int32)]


class Layout(ctypes.Structure):
    """i8c_layout: the shared- and tensor-memory layout of a plan's kernel."""
    _fields_ = [(n, ctypes.c_int32) for n in (
        "kernel_variant", "cta_group", "block_n", "smem_bytes", "tmem_cols", "chunk_slices", "num_chunks",
        "flat_tiles", "tile_px", "halo_rows", "halo_cw", "positions", "plane_bytes", "halo_bytes", "halo_stages",
        "off_staging", "staging_slots", "staging_bytes", "off_filter", "filter_stages", "filter_run",
        "filter_stage_bytes", "off_out", "off_bar", "bar_bytes")] + [("phase_off", ctypes.c_int32 * 9)] + [
        (n, ctypes.c_int32) for n in ("tma_halo", "x8_slots", "off_x8", "x8_bytes", "box_w", "box_h",
            "gather_stages", "gather_off_a", "gather_stage_a", "gather_off_b", "gather_stage_b",
            "gather_off_staging", "gather_staging_slots", "gather_staging_bytes", "gather_off_bar",
            "subtiles")]

    def asdict(self):
        d = {n: getattr(self, n) for n, _ in self._fields_}
        d["phase_off"] = list(self.phase_off)
        return d


class TuneEntry(ctypes.Structure):
    """i8c_tune_entry: one candidate of i8c_plan_autotune."""
    _fields_ = [("options", Options), ("status", ctypes.c_int32), ("us", ctypes.c_float)]


class PlanInfo(ctypes.Structure):
    _fields_ = [("P", ctypes.c_int32), ("Q", ctypes.c_int32), ("M", ctypes.c_int64),
                ("gemm_n", ctypes.c_int32), ("gemm_k", ctypes.c_int32),
                ("block_m", ctypes.c_int32), ("block_n", ctypes.c_int32),
                ("num_tiles", ctypes.c_int32), ("num_ctas", ctypes.c_int32),
                ("num_chunks", ctypes.c_int32), ("chunk_slices", ctypes.c_int32),
                ("acc_buffers", ctypes.c_int32), ("smem_bytes", ctypes.c_int32),
                ("kernels_per_run", ctypes.c_int32), ("ops", ctypes.c_int64),
                ("workspace_bytes", ctypes.c_int64), ("kernel_variant", ctypes.c_int32),
                ("halo_staging", ctypes.c_int32), ("filter_run", ctypes.c_int32),
                ("filter_stages", ctypes.c_int32), ("tail_split", ctypes.c_int32),
                ("work_units", ctypes.c_int32), ("tail_halves", ctypes.c_int32), ("flat_tiles", ctypes.c_int32),
                ("filter_resident", ctypes.c_int32)]

    def asdict(self):
        return {n: getattr(self, n) for n, _ in self._fields_}


def _load() -> ctypes.CDLL:
    if not os.path.exists(LIB_PATH):
        raise ImportError(f"{LIB_PATH} is not built; run int8_implicit_gemm_gb300/build_lib.py "
                          "(or __graft_entry__.build()) first -- there is no fallback path")
    lib = ctypes.CDLL(LIB_PATH)
    P, I32, I64, F = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_float
    S = ctypes.POINTER(ConvShape)
    sig = {
        "i8c_output_size": [S, ctypes.POINTER(I32), ctypes.POINTER(I32)],
        "i8c_supported": [S],
        "i8c_conv2d_fprop": [P, P, P, S, F, P],
        "i8c_conv2d_fprop_acc": [P, P, P, S, P],
        "i8c_conv2d_fprop_noalloc": [P, P, P, S, F, P],
        "i8c_conv2d_fprop_f32": [P, P, P, P, S, P],
        "i8c_last_device_status": [P],
        "i8c_debug_set_oneshot": [I32, I32],
        "i8c_plan_create": [S, ctypes.POINTER(Options), ctypes.POINTER(P)],
        "i8c_plan_run": [P, P, P, P, F, P],
        "i8c_plan_run_ex": [P, P, P, P, F, ctypes.POINTER(Epilogue), P],
        "i8c_plan_set_filter": [P, P, P],
        "i8c_plan_run_prepacked": [P, P, P, F, P],
        "i8c_plan_run_prepacked_ex": [P, P, P, F, ctypes.POINTER(Epilogue), P],
        "i8c_conv2d_fprop_ex": [P, P, P, S, F, ctypes.POINTER(Epilogue), P],
        "i8c_plan_run_acc": [P, P, P, P, P],
        "i8c_plan_run_host": [P, P, P, P, F, P],
        "i8c_plan_run_host_pipelined": [P, P, P, P, P, I32, P],
        "i8c_plan_status": [P, P],
        "i8c_plan_get_info": [P, ctypes.POINTER(PlanInfo)],
        "i8c_plan_layout": [S, ctypes.POINTER(Options), I32, ctypes.POINTER(Layout)],
        "i8c_plan_get_layout": [P, ctypes.POINTER(Layout)],
        "i8c_plan_kernel_time": [P, ctypes.POINTER(ctypes.c_double), ctypes.POINTER(I64)],
        "i8c_plan_trace": [P, P, I64],
        "i8c_plan_destroy": [P],
        "i8c_plan_autotune": [S, P, P, P, F, I32, P, ctypes.POINTER(Options), ctypes.POINTER(F),
                              ctypes.POINTER(TuneEntry), I32, ctypes.POINTER(I32)],
        "i8c_pack_nchw_to_ncxhwx32": [P, P, I32, I32, I32, I32, P],
        "i8c_unpack_ncxhwx32_to_nchw": [P, P, I32, I32, I32, I32, P],
        "i8c_pack_kcrs_to_cxrskx32": [P, P, I32, I32, I32, I32, P],
        "i8c_unpack_cxrskx32_to_kcrs": [P, P, I32, I32, I32, I32, P],
    }
    for name, args in sig.items():
        fn = getattr(lib, name)
        fn.argtypes = args
        fn.restype = ctypes.c_int
    lib.i8c_probe_mma_f16.argtypes = [I32, I32, I32, I32, I32, P, ctypes.POINTER(F), P]
    lib.i8c_probe_mma_f16.restype = ctypes.c_int
    lib.i8c_probe_imma_s8.argtypes = [I32, I32, I32, P, P, ctypes.POINTER(F), P]
    lib.i8c_probe_imma_s8.restype = ctypes.c_int
    lib.i8c_probe_mma_f8.argtypes = [I32, I32, I32, P, ctypes.POINTER(F), P]
    lib.i8c_probe_mma_f8.restype = ctypes.c_int
    lib.i8c_probe_l2_ingress.argtypes = [P, I64, I32, I32, I32, I32, P, ctypes.POINTER(F), P]
    lib.i8c_probe_l2_ingress.restype = ctypes.c_int
    lib.i8c_status_string.argtypes = [ctypes.c_int]
    lib.i8c_status_string.restype = ctypes.c_char_p
    lib.i8c_launch_count.argtypes = []
    lib.i8c_launch_count.restype = I64
    lib.i8c_oneshot_cached_plans.argtypes = []
    lib.i8c_oneshot_cached_plans.restype = I64
    return lib


lib = _load()


def status_string(status: int) -> str:
    return lib.i8c_status_string(int(status)).decode()


def _check(status: int, where: str) -> None:
    if status != I8C_OK:
        raise I8ConvError(status, where)


def _ptr(t) -> int:
    """Raw address of a tensor's data (torch tensor) or of a numpy array."""
    if hasattr(t, "data_ptr"):
        return t.data_ptr()
    return t.ctypes.data


def _stream(stream) -> int:
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if hasattr(stream, "cuda_stream"):
        return stream.cuda_stream
    return int(stream)


def launch_count() -> int:
    return int(lib.i8c_launch_count())


def i8c_output_size(shape):
    P, Q = ctypes.c_int32(), ctypes.c_int32()
    _check(lib.i8c_output_size(ctypes.byref(ConvShape.of(shape)), ctypes.byref(P), ctypes.byref(Q)),
           "i8c_output_size")
    return P.value, Q.value


def i8c_supported(shape) -> int:
    """Status code of the argument check (0 = supported)."""
    return lib.i8c_supported(ctypes.byref(ConvShape.of(shape)))


def i8c_conv2d_fprop(x, f, y, shape, alpha: float, stream=None) -> None:
    _check(lib.i8c_conv2d_fprop(_ptr(x), _ptr(f), _ptr(y), ctypes.byref(ConvShape.of(shape)),
                                ctypes.c_float(alpha), _stream(stream)), "i8c_conv2d_fprop")


def i8c_conv2d_fprop_ex(x, f, y, shape, alpha: float, alpha_k=None, bias=None, relu: bool = False,
                        stream=None) -> None:
    """One-shot run with the per-output-channel epilogue (alpha_k, bias: CUDA
    float32 tensors of K values or None)."""
    ep = Epilogue(None if alpha_k is None else _ptr(alpha_k), None if bias is None else _ptr(bias), int(bool(relu)))
    _check(lib.i8c_conv2d_fprop_ex(_ptr(x), _ptr(f), _ptr(y), ctypes.byref(ConvShape.of(shape)),
                                   ctypes.c_float(alpha), ctypes.byref(ep), _stream(stream)), "i8c_conv2d_fprop_ex")


def i8c_conv2d_fprop_acc(x, f, acc, shape, stream=None) -> None:
    _check(lib.i8c_conv2d_fprop_acc(_ptr(x), _ptr(f), _ptr(acc), ctypes.byref(ConvShape.of(shape)),
                                    _stream(stream)), "i8c_conv2d_fprop_acc")


def i8c_conv2d_fprop_noalloc(x, f, y, shape, alpha: float, stream=None) -> None:
    """The convolution without any device allocation: scratch lives in the
    library's fixed static device array (see include/i8conv.h)."""
    _check(lib.i8c_conv2d_fprop_noalloc(_ptr(x), _ptr(f), _ptr(y), ctypes.byref(ConvShape.of(shape)),
                                        ctypes.c_float(alpha), _stream(stream)), "i8c_conv2d_fprop_noalloc")


def i8c_last_device_status(stream=None) -> int:
    """Synchronise the stream and return (and clear) the device status of the
    one-shot calls made on it (and of the no-allocation entry point)."""
    return lib.i8c_last_device_status(_stream(stream))


def i8c_oneshot_cached_plans() -> int:
    return lib.i8c_oneshot_cached_plans()


def i8c_debug_set_oneshot(debug_flags: int = 0, wait_timeout_us: int = 0) -> None:
    _check(lib.i8c_debug_set_oneshot(debug_flags, wait_timeout_us), "i8c_debug_set_oneshot")


def make_options(**kw) -> "Options":
    """i8c_options from keyword arguments (the Plan constructor's names)."""
    o = Options()
    for k, v in kw.items():
        if k not in dict(Options._fields_):
            raise TypeError(f"unknown plan option {k}")
        setattr(o, k, int(v))
    return o


def i8c_plan_layout(shape, num_sms: int = 152, **options) -> dict:
    """The layout a plan of `shape` with these options would get on a GPU of
    num_sms SMs, computed on the host alone (no GPU needed)."""
    out = Layout()
    _check(lib.i8c_plan_layout(ctypes.byref(ConvShape.of(shape)), ctypes.byref(make_options(**options)), num_sms,
                               ctypes.byref(out)), "i8c_plan_layout")
    return out.asdict()


def i8c_plan_autotune(x, f, y, shape, alpha: float, iters: int = 10, stream=None):
    """Time the candidate plans of `shape` on these tensors (i8c_plan_autotune).
    Returns (options, us, entries): the fastest candidate's plan options as a
    dict of Plan keyword arguments, its mean time per run in microseconds, and
    every candidate as (options dict, status, us).  y holds the chosen plan's
    output afterwards."""
    best, best_us = Options(), ctypes.c_float()
    cap = 64
    entries, n = (TuneEntry * cap)(), ctypes.c_int32()
    _check(lib.i8c_plan_autotune(ctypes.byref(ConvShape.of(shape)), _ptr(x), _ptr(f), _ptr(y), ctypes.c_float(alpha),
                                 int(iters), _stream(stream), ctypes.byref(best), ctypes.byref(best_us), entries, cap,
                                 ctypes.byref(n)), "i8c_plan_autotune")

    def opts(o):
        return {name: getattr(o, name) for name, _ in Options._fields_}

    return opts(best), best_us.value, [(opts(e.options), e.status, e.us) for e in entries[:n.value]]


def i8c_conv2d_fprop_f32(x, w, bias, y, shape, stream=None) -> None:
    """fp32 direct convolution (NCHW / KCRS, optional bias) on the SIMT cores."""
    _check(lib.i8c_conv2d_fprop_f32(_ptr(x), _ptr(w), None if bias is None else _ptr(bias), _ptr(y),
                                    ctypes.byref(ConvShape.of(shape)), _stream(stream)), "i8c_conv2d_fprop_f32")


def conv2d_fprop_f32(x, w, shape, bias=None, out=None, stream=None):
    """Convenience wrapper: allocate the NCHW fp32 output with torch and run."""
    import torch
    s = ConvShape.of(shape)
    P, Q = i8c_output_size(s)
    if out is None:
        out = torch.empty((s.N, s.K, P, Q), dtype=torch.float32, device=x.device)
    i8c_conv2d_fprop_f32(x, w, bias, out, s, stream)
    return out


def i8c_pack_nchw_to_ncxhwx32(src, dst, N, C, H, W, stream=None) -> None:
    _check(lib.i8c_pack_nchw_to_ncxhwx32(_ptr(src), _ptr(dst), N, C, H, W, _stream(stream)), "pack")


def i8c_unpack_ncxhwx32_to_nchw(src, dst, N, C, H, W, stream=None) -> None:
    _check(lib.i8c_unpack_ncxhwx32_to_nchw(_ptr(src), _ptr(dst), N, C, H, W, _stream(stream)), "unpack")


def i8c_pack_kcrs_to_cxrskx32(src, dst, K, C, R, S, stream=None) -> None:
    _check(lib.i8c_pack_kcrs_to_cxrskx32(_ptr(src), _ptr(dst), K, C, R, S, _stream(stream)), "pack")


def i8c_unpack_cxrskx32_to_kcrs(src, dst, K, C, R, S, stream=None) -> None:
    _check(lib.i8c_unpack_cxrskx32_to_kcrs(_ptr(src), _ptr(dst), K, C, R, S, _stream(stream)), "unpack")


def i8c_probe_mma_f16(n: int, a_swizzled: int, num_ctas: int, iters: int, loop_mode: int = 0, stream=None):
    """Tensor-core probe (include/i8conv_probe.h): returns (per-CTA cycles array
    [num_ctas, 3] = issue cycles, completion cycles, ok flag; elapsed ms)."""
    import torch
    buf = torch.zeros(3 * num_ctas, dtype=torch.int64, device="cuda")
    ms = ctypes.c_float()
    _check(lib.i8c_probe_mma_f16(n, int(a_swizzled), loop_mode, num_ctas, iters, buf.data_ptr(), ctypes.byref(ms),
                                 _stream(stream)), "i8c_probe_mma_f16")
    return buf.cpu().numpy().reshape(num_ctas, 3), ms.value


def i8c_probe_imma_s8(num_ctas: int, warps_per_cta: int, iters: int, stream=None):
    """Warp-level s8 IMMA probe: (per-CTA cycles [num_ctas, 3], elapsed ms)."""
    import torch
    buf = torch.zeros(3 * num_ctas, dtype=torch.int64, device="cuda")
    sink = torch.zeros(1, dtype=torch.int32, device="cuda")
    ms = ctypes.c_float()
    _check(lib.i8c_probe_imma_s8(num_ctas, warps_per_cta, iters, buf.data_ptr(), sink.data_ptr(), ctypes.byref(ms),
                                 _stream(stream)), "i8c_probe_imma_s8")
    return buf.cpu().numpy().reshape(num_ctas, 3), ms.value


def i8c_probe_l2_ingress(src, region_bytes: int, chunk_bytes: int, mode: int, num_ctas: int, iters: int,
                         stream=None):
    """L2 -> shared memory read-rate probe over the device tensor `src`:
    (per-CTA [cycles, bytes, ok] as [num_ctas, 3], elapsed ms)."""
    import torch
    buf = torch.zeros(3 * num_ctas, dtype=torch.int64, device="cuda")
    ms = ctypes.c_float()
    _check(lib.i8c_probe_l2_ingress(src.data_ptr(), region_bytes, chunk_bytes, mode, num_ctas, iters, buf.data_ptr(),
                                    ctypes.byref(ms), _stream(stream)), "i8c_probe_l2_ingress")
    return buf.cpu().numpy().reshape(num_ctas, 3), ms.value


def i8c_probe_mma_f8(n: int, num_ctas: int, iters: int, stream=None):
    """tcgen05 kind::f8f6f4 (e4m3) probe: (per-CTA cycles [num_ctas, 3], elapsed ms)."""
    import torch
    buf = torch.zeros(3 * num_ctas, dtype=torch.int64, device="cuda")
    ms = ctypes.c_float()
    _check(lib.i8c_probe_mma_f8(n, num_ctas, iters, buf.data_ptr(), ctypes.byref(ms), _stream(stream)),
           "i8c_probe_mma_f8")
    return buf.cpu().numpy().reshape(num_ctas, 3), ms.value


class Plan:
    """A validated convolution plan on the current CUDA device (i8c_plan_*)."""

    def __init__(self, shape, block_n=0, num_ctas=0, max_chunk_slices=0, wait_timeout_us=0,
                 host_staging=False, debug_flags=0, timing_events=0, kernel_variant=0, halo_loads=0, tail_split=0,
                 tile_shape=0, fused_filter=0, tile_px=0, filter_run=0):
        self.shape = ConvShape.of(shape)
        opts = Options(block_n, num_ctas, max_chunk_slices, wait_timeout_us, int(host_staging), debug_flags,
                       timing_events, kernel_variant, halo_loads, tail_split, tile_shape, fused_filter, tile_px,
                       filter_run)
        h = ctypes.c_void_p()
        _check(lib.i8c_plan_create(ctypes.byref(self.shape), ctypes.byref(opts), ctypes.byref(h)),
               "i8c_plan_create")
        self.handle = h
        info = PlanInfo()
        _check(lib.i8c_plan_get_info(self.handle, ctypes.byref(info)), "i8c_plan_get_info")
        self.info = info.asdict()

    def run(self, x, f, y, alpha: float, stream=None, alpha_k=None, bias=None, relu: bool = False) -> None:
        """y = clamp(rint(alpha * acc)); with alpha_k / bias (CUDA float32 tensors
        of K values) or relu, the per-output-channel epilogue (i8c_plan_run_ex)."""
        if alpha_k is None and bias is None and not relu:
            _check(lib.i8c_plan_run(self.handle, _ptr(x), _ptr(f), _ptr(y), ctypes.c_float(alpha), _stream(stream)),
                   "i8c_plan_run")
            return
        ep = Epilogue(None if alpha_k is None else _ptr(alpha_k), None if bias is None else _ptr(bias), int(bool(relu)))
        _check(lib.i8c_plan_run_ex(self.handle, _ptr(x), _ptr(f), _ptr(y), ctypes.c_float(alpha), ctypes.byref(ep),
                                   _stream(stream)), "i8c_plan_run_ex")

    def set_filter(self, f, stream=None) -> None:
        """Weight prepacking: convert the filter once into the plan's operand
        copy (i8c_plan_set_filter), for run_prepacked."""
        _check(lib.i8c_plan_set_filter(self.handle, _ptr(f), _stream(stream)), "i8c_plan_set_filter")

    def run_prepacked(self, x, y, alpha: float, stream=None, alpha_k=None, bias=None, relu: bool = False) -> None:
        """As run, with the filter given to set_filter (no conversion launch)."""
        if alpha_k is None and bias is None and not relu:
            _check(lib.i8c_plan_run_prepacked(self.handle, _ptr(x), _ptr(y), ctypes.c_float(alpha), _stream(stream)),
                   "i8c_plan_run_prepacked")
            return
        ep = Epilogue(None if alpha_k is None else _ptr(alpha_k), None if bias is None else _ptr(bias), int(bool(relu)))
        _check(lib.i8c_plan_run_prepacked_ex(self.handle, _ptr(x), _ptr(y), ctypes.c_float(alpha), ctypes.byref(ep),
                                             _stream(stream)), "i8c_plan_run_prepacked_ex")

    def run_acc(self, x, f, acc, stream=None) -> None:
        _check(lib.i8c_plan_run_acc(self.handle, _ptr(x), _ptr(f), _ptr(acc), _stream(stream)), "i8c_plan_run_acc")

    def run_host(self, x_host, f_host, y_host, alpha: float, stream=None) -> None:
        _check(lib.i8c_plan_run_host(self.handle, _ptr(x_host), _ptr(f_host), _ptr(y_host), ctypes.c_float(alpha),
                                     _stream(stream)), "i8c_plan_run_host")

    def run_host_pipelined(self, x_hosts, f_hosts, y_hosts, alphas, stream=None) -> None:
        """len(x_hosts) end-to-end runs on pinned host tensors, the copies of
        neighbouring runs overlapped (plan created with host_staging=2)."""
        n = len(x_hosts)
        if not (len(f_hosts) == len(y_hosts) == len(alphas) == n):
            raise ValueError("one x, f, y and alpha per run")
        arr = ctypes.c_void_p * max(1, n)
        xa, fa, ya = arr(*[_ptr(t) for t in x_hosts]), arr(*[_ptr(t) for t in f_hosts]), arr(*[_ptr(t) for t in y_hosts])
        al = (ctypes.c_float * max(1, n))(*[float(a) for a in alphas])
        _check(lib.i8c_plan_run_host_pipelined(self.handle, xa, fa, ya, al, n, _stream(stream)),
               "i8c_plan_run_host_pipelined")

    def kernel_time(self):
        """(summed ms, launches) of the convolution kernels timed since the last call."""
        ms, n = ctypes.c_double(), ctypes.c_int64()
        _check(lib.i8c_plan_kernel_time(self.handle, ctypes.byref(ms), ctypes.byref(n)), "i8c_plan_kernel_time")
        return ms.value, n.value

    def layout(self) -> dict:
        """The shared- and tensor-memory layout of this plan's kernel."""
        out = Layout()
        _check(lib.i8c_plan_get_layout(self.handle, ctypes.byref(out)), "i8c_plan_get_layout")
        return out.asdict()

    def trace(self):
        """The trace of a plan created with I8C_DEBUG_TRACE, shape (8, 4, 512):
        [role][event][step] clock64 values of CTA 0 for roles 0-3 (MMA issuer,
        filter TMA, activation producer, epilogue); rows 4-7 are written only
        by pipeline-analysis builds."""
        import numpy as np
        out = np.zeros(32 * 512, dtype=np.int64)
        _check(lib.i8c_plan_trace(self.handle, out.ctypes.data, out.size), "i8c_plan_trace")
        return out.reshape(8, 4, 512)

    def status(self, stream=None) -> int:
        """Synchronise and return (and clear) the device status word."""
        return lib.i8c_plan_status(self.handle, _stream(stream))

    def destroy(self) -> None:
        if self.handle:
            _check(lib.i8c_plan_destroy(self.handle), "i8c_plan_destroy")
            self.handle = None

    def __del__(self):
        try:
            if getattr(self, "handle", None):
                lib.i8c_plan_destroy(self.handle)
        except Exception:
            pass


def output_nbytes(shape) -> int:
    s = ConvShape.of(shape)
    P, Q = i8c_output_size(s)
    return s.N * s.K * P * Q


def conv2d_fprop(x, f, shape, alpha: float, out=None, stream=None):
    """Convenience wrapper: allocate the NCxHWx<32> int8 output with torch and run."""
    import torch
    s = ConvShape.of(shape)
    P, Q = i8c_output_size(s)
    if out is None:
        out = torch.empty((s.N, s.K // 32, P, Q, 32), dtype=torch.int8, device=x.device)
    i8c_conv2d_fprop(x, f, out, s, alpha, stream)
    return out
