"""The C-ABI library on a machine without a GPU: it loads, exports every entry
point its header declares, and its host-side argument checks behave as
documented.  No compute call is made here."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def ext():
    import __graft_entry__
    __graft_entry__.build()
    import int8_implicit_gemm_gb300 as ext
    return ext


def _declared(header):
    text = open(os.path.join(ROOT, "include", header)).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(i8c_[a-z0-9_]+)\s*\(", text)))


def test_every_declared_symbol_is_exported(ext):
    headers = [h for h in os.listdir(os.path.join(ROOT, "include")) if h.endswith(".h")]
    assert headers
    lib = ctypes.CDLL(ext.LIB_PATH)
    for h in headers:
        names = _declared(h)
        assert names, h
        for name in names:
            assert hasattr(lib, name), f"{name} declared in {h} but not exported"


def test_status_strings(ext):
    assert ext.status_string(0) == "ok"
    assert "aligned" in ext.status_string(ext.I8C_ERR_MISALIGNED)
    assert ext.status_string(99) == "unknown status"


def test_output_size_page4(ext):
    # the 5x9 dilated layer of the kernel-benchmark trace: 508 x 496
    assert ext.i8c_output_size((8, 32, 512, 512, 64, 5, 9, 2, 4, 1, 1, 2, 3)) == (508, 496)
    assert ext.i8c_output_size((32, 128, 112, 112, 256, 3, 3, 1, 1, 2, 2, 1, 1)) == (56, 56)


@pytest.mark.parametrize("shape,status", [
    ((1, 32, 16, 16, 32, 3, 3, 1, 1, 1, 1, 1, 1), 0),
    ((1, 48, 16, 16, 32, 3, 3, 1, 1, 1, 1, 1, 1), 2),       # C not a multiple of 32
    ((1, 32, 16, 16, 40, 3, 3, 1, 1, 1, 1, 1, 1), 2),       # K not a multiple of 32
    ((1, 32, 2, 2, 32, 5, 5, 0, 0, 1, 1, 1, 1), 2),         # filter larger than the padded input
    ((0, 32, 16, 16, 32, 3, 3, 1, 1, 1, 1, 1, 1), 1),       # empty batch
    ((1, 32, 16, 16, 32, 3, 3, -1, 1, 1, 1, 1, 1), 1),      # negative padding
    ((1, 32, 16, 16, 32, 3, 3, 1, 1, 0, 1, 1, 1), 1),       # zero stride
    ((1, 32, 16, 16, 32, 3, 3, 1, 1, 1, 1, 1, 0), 1),       # zero dilation
    ((1, 4096, 64, 64, 32, 7, 7, 3, 3, 1, 1, 1, 1), 4),     # C*R*S*2^14 >= 2^31
])
def test_supported(ext, shape, status):
    assert ext.i8c_supported(shape) == status


def test_no_cpu_fallback(ext):
    """Without a usable device the library refuses to run instead of computing on the host."""
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    with pytest.raises(ext.I8ConvError) as ei:
        ext.Plan((1, 32, 16, 16, 32, 3, 3, 1, 1, 1, 1, 1, 1))
    assert ei.value.status in (ext.I8C_ERR_NO_DEVICE, ext.I8C_ERR_CUDA)


def test_null_pointers_rejected(ext):
    st = ext.lib.i8c_conv2d_fprop(None, None, None, ctypes.byref(ext.ConvShape.of(
        (1, 32, 16, 16, 32, 3, 3, 1, 1, 1, 1, 1, 1))), ctypes.c_float(1.0), None)
    assert st == ext.I8C_ERR_INVALID_ARG


def test_prepacked_argument_checks(ext):
    """Weight prepacking refuses a missing plan, filter or buffer before
    touching a device."""
    a = ctypes.c_void_p(16)
    assert ext.lib.i8c_plan_set_filter(None, a, None) == ext.I8C_ERR_INVALID_ARG
    assert ext.lib.i8c_plan_run_prepacked(None, a, a, ctypes.c_float(1.0), None) == ext.I8C_ERR_INVALID_ARG
    assert ext.lib.i8c_plan_run_prepacked_ex(None, a, a, ctypes.c_float(1.0), None, None) == ext.I8C_ERR_INVALID_ARG


def test_autotune_argument_checks(ext):
    """The tuner rejects bad arguments on the host, before touching a device."""
    shape = ctypes.byref(ext.ConvShape.of((1, 32, 16, 16, 32, 3, 3, 1, 1, 1, 1, 1, 1)))
    best, us, n = ext.Options(), ctypes.c_float(), ctypes.c_int32()
    buf = ctypes.create_string_buffer(64)
    a = (ctypes.addressof(buf) + 15) & ~15
    call = ext.lib.i8c_plan_autotune
    assert call(shape, None, a, a, 1.0, 4, None, ctypes.byref(best), ctypes.byref(us), None, 0, None) == \
        ext.I8C_ERR_INVALID_ARG
    assert call(shape, a, a, a, 1.0, 0, None, ctypes.byref(best), ctypes.byref(us), None, 0, None) == \
        ext.I8C_ERR_INVALID_ARG                                                  # iters < 1
    assert call(shape, a, a, a, 1.0, 4, None, ctypes.byref(best), ctypes.byref(us), None, 3, ctypes.byref(n)) == \
        ext.I8C_ERR_INVALID_ARG                                                  # entries NULL, max_entries > 0
    assert call(shape, a + 1, a, a, 1.0, 4, None, ctypes.byref(best), ctypes.byref(us), None, 0, None) == \
        ext.I8C_ERR_MISALIGNED
    bad = ctypes.byref(ext.ConvShape.of((1, 48, 16, 16, 32, 3, 3, 1, 1, 1, 1, 1, 1)))
    assert call(bad, a, a, a, 1.0, 4, None, ctypes.byref(best), ctypes.byref(us), None, 0, None) == \
        ext.I8C_ERR_UNSUPPORTED                                                  # C not a multiple of 32


@pytest.mark.parametrize("opts", [
    dict(block_n=48), dict(block_n=512), dict(num_ctas=-1), dict(max_chunk_slices=33), dict(wait_timeout_us=-5),
    dict(timing_events=70000), dict(kernel_variant=7), dict(halo_loads=4), dict(tail_split=4), dict(tile_shape=4),
    dict(fused_filter=4), dict(tile_px=20), dict(tile_px=272), dict(tile_px=8), dict(filter_run=33),
], ids=lambda o: ",".join(f"{k}={v}" for k, v in o.items()))
def test_plan_options_rejected_on_the_host(ext, opts):
    """Out-of-range plan options are refused before any device is touched."""
    fields = {n: 0 for n, _ in ext.Options._fields_}
    fields.update(opts)
    o = ext.Options(**fields)
    h = ctypes.c_void_p()
    shape = ctypes.byref(ext.ConvShape.of((1, 32, 16, 16, 32, 3, 3, 1, 1, 1, 1, 1, 1)))
    assert ext.lib.i8c_plan_create(shape, ctypes.byref(o), ctypes.byref(h)) == ext.I8C_ERR_INVALID_ARG
    assert not h.value


def test_f32_direct_argument_checks(ext):
    """The fp32 entry point's host-side checks: null, misaligned, invalid and
    unsupported shapes; a valid call without a GPU fails with a device error."""
    buf = ctypes.create_string_buffer(64)
    a = (ctypes.addressof(buf) + 15) & ~15
    f = ext.lib.i8c_conv2d_fprop_f32
    good = ctypes.byref(ext.ConvShape.of((1, 3, 8, 8, 4, 3, 3, 1, 1, 1, 1, 1, 1)))
    assert f(None, a, None, a, good, None) == ext.I8C_ERR_INVALID_ARG
    assert f(a, a, None, a, None, None) == ext.I8C_ERR_INVALID_ARG
    assert f(a + 2, a, None, a, good, None) == ext.I8C_ERR_MISALIGNED
    assert f(a, a, a + 1, a, good, None) == ext.I8C_ERR_MISALIGNED            # bias misaligned
    assert f(a, a, None, a, ctypes.byref(ext.ConvShape.of((1, 3, 2, 2, 4, 5, 5, 0, 0, 1, 1, 1, 1))),
             None) == ext.I8C_ERR_UNSUPPORTED                                    # empty output
    assert f(a, a, None, a, ctypes.byref(ext.ConvShape.of((1, 3, 8, 8, 4, 3, 3, 1, 1, 0, 1, 1, 1))),
             None) == ext.I8C_ERR_INVALID_ARG                                    # zero stride
    assert f(a, a, None, a, ctypes.byref(ext.ConvShape.of((70000, 3, 8, 8, 4, 3, 3, 1, 1, 1, 1, 1, 1))),
             None) == ext.I8C_ERR_UNSUPPORTED                                    # batch past the grid's y extent
    import torch
    if not torch.cuda.is_available():
        assert f(a, a, None, a, good, None) in (ext.I8C_ERR_NO_DEVICE, ext.I8C_ERR_CUDA)


def test_noalloc_argument_checks(ext):
    """The no-allocation entry point refuses bad arguments on the host."""
    buf = ctypes.create_string_buffer(64)
    a = (ctypes.addressof(buf) + 15) & ~15
    f = ext.lib.i8c_conv2d_fprop_noalloc
    good = ctypes.byref(ext.ConvShape.of((1, 32, 16, 16, 32, 3, 3, 1, 1, 1, 1, 1, 1)))
    assert f(None, a, a, good, ctypes.c_float(1.0), None) == ext.I8C_ERR_INVALID_ARG
    assert f(a + 1, a, a, good, ctypes.c_float(1.0), None) == ext.I8C_ERR_MISALIGNED
    assert f(a, a, a, ctypes.byref(ext.ConvShape.of((1, 48, 16, 16, 32, 3, 3, 1, 1, 1, 1, 1, 1))),
             ctypes.c_float(1.0), None) == ext.I8C_ERR_UNSUPPORTED


def test_build_flavour_stamp(tmp_path, monkeypatch):
    """The build script rebuilds when the requested flavour (release or
    pipeline trace) differs from the one the library was built with."""
    import importlib.util
    spec = importlib.util.spec_from_file_location("bl", os.path.join(ROOT, "int8_implicit_gemm_gb300", "build_lib.py"))
    bl = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(bl)
    lib = tmp_path / "libi8conv.so"
    stamp = tmp_path / "flavour"
    lib.write_bytes(b"x")
    monkeypatch.setattr(bl, "LIB", str(lib))
    monkeypatch.setattr(bl, "STAMP", str(stamp))
    monkeypatch.setattr(bl, "_deps", lambda: [])
    assert not bl.up_to_date(False)                   # no stamp yet
    stamp.write_text("release")
    assert bl.up_to_date(False) and not bl.up_to_date(True)
    stamp.write_text("pipeline-trace")
    assert bl.up_to_date(True) and not bl.up_to_date(False)


@pytest.mark.parametrize("ctype,cls_name", [("i8c_conv_shape", "ConvShape"), ("i8c_options", "Options"),
                                            ("i8c_plan_info", "PlanInfo"), ("i8c_epilogue", "Epilogue"),
                                            ("i8c_tune_entry", "TuneEntry")])
def test_binding_structs_match_header(ext, tmp_path, ctype, cls_name):
    """The binding's ctypes structures have the header's size and field offsets
    (compiled with the host C compiler against include/i8conv.h)."""
    import shutil
    import subprocess
    if shutil.which("gcc") is None:
        pytest.skip("no host C compiler")
    cls = getattr(ext, cls_name)
    fields = [n for n, _ in cls._fields_]
    lines = [f'  printf("size %zu\\n", sizeof({ctype}));']
    lines += [f'  printf("{n} %zu\\n", offsetof({ctype}, {n}));' for n in fields]
    src = tmp_path / "abi.c"
    src.write_text('#include <stddef.h>\n#include <stdio.h>\n#include "i8conv.h"\nint main(void) {\n'
                   + "\n".join(lines) + "\n  return 0;\n}\n")
    exe = tmp_path / "abi"
    cuda_inc = os.path.join(os.environ.get("CUDA_HOME", "/usr/local/cuda"), "include")
    subprocess.run(["gcc", "-std=c99", "-I", os.path.join(ROOT, "include"), "-I", cuda_inc, str(src), "-o", str(exe)],
                   check=True)
    out = dict(line.split() for line in subprocess.run([str(exe)], check=True, capture_output=True,
                                                         text=True).stdout.splitlines())
    assert int(out["size"]) == ctypes.sizeof(cls)
    for n in fields:
        assert int(out[n]) == getattr(cls, n).offset, n
