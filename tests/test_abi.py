"""The C ABI without a GPU: the library builds, loads, exports every
function include/tqd.h declares, names its statuses, and refuses bad
configurations before touching a device."""
import ctypes
import os
import re

import pytest

import synth
import token_quantized_decode_gb300 as tqd
from token_quantized_decode_gb300 import _lib
from token_quantized_decode_gb300 import build as tqd_build

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include", "tqd.h")


@pytest.fixture(scope="module")
def L():
    tqd_build.build()
    return _lib.lib()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return re.findall(r"^\s*(?:const\s+char\s*\*|int32_t|void|size_t)\s+(tqd_\w+)\s*\(", text, flags=re.M)


def test_every_declared_symbol_is_exported(L):
    names = declared_functions()
    assert len(names) >= 20
    for n in names:
        assert hasattr(L, n), f"{n} declared in tqd.h but not exported"
    assert set(names) == set(_lib.exported_symbols())


def test_status_names_need_no_device(L):
    for i, n in enumerate(_lib.STATUS_NAMES):
        assert tqd.tqd_status_name(i) == n
    assert tqd.tqd_status_name(-1) == "TQD_UNKNOWN_STATUS"
    assert tqd.tqd_status_name(1000) == "TQD_UNKNOWN_STATUS"


def test_config_struct_layout_matches_header(L):
    # 11 int32 / float fields before max_seq, then max_seq, max_batch, schedule, kv_type
    assert ctypes.sizeof(_lib.tqd_config) == 15 * 4
    assert ctypes.sizeof(_lib.tqd_layer_weights) == 11 * ctypes.sizeof(ctypes.c_void_p)
    assert ctypes.sizeof(_lib.tqd_host_weights) == 4 * ctypes.sizeof(ctypes.c_void_p)


def test_bad_configs_are_refused_before_any_device_work(L):
    m = synth.make_model(synth.TINY, 0)
    w = tqd.make_host_weights(m)
    bad = [("head_dim", 96), ("n_kv_heads", 3), ("max_seq", 0), ("max_batch", 0), ("schedule", 7),
           ("hidden", 250), ("weight_type", 5)]
    for field, val in bad:
        c = tqd.make_config(synth.TINY, 16)
        setattr(c, field, val)
        with pytest.raises(tqd.TQDError) as ei:
            tqd.tqd_create(c, w)
        assert ei.value.name == "TQD_ERR_UNSUPPORTED_CONFIG", (field, ei.value)
    # every mismatched field is named in one refusal
    c = tqd.make_config(synth.TINY, 16)
    c.head_dim = 96
    c.max_seq = 0
    with pytest.raises(tqd.TQDError) as ei:
        tqd.tqd_create(c, w)
    msg = str(ei.value)
    assert "head_dim" in msg and "max_seq" in msg


def test_null_arguments_are_refused(L):
    assert L.tqd_create(None, None, None, None) == _lib.TQD_ERR_BAD_ARG
    assert L.tqd_create_synthetic(None, 0, None, None) == _lib.TQD_ERR_BAD_ARG
    assert L.tqd_export_weights(None, None) == _lib.TQD_ERR_BAD_ARG
    assert L.tqd_decode_step(None, 0, 0, 0, None) == _lib.TQD_ERR_BAD_ARG
    assert L.tqd_generate(None, 0, 0, 1, None) == _lib.TQD_ERR_BAD_ARG
    assert L.tqd_phase_count(None, None) == _lib.TQD_ERR_BAD_ARG
    assert L.tqd_op_argmax(None, 0, None, None, None) == _lib.TQD_ERR_BAD_ARG
    assert L.tqd_op_q8_0_matvec(None, 4, 96, None, None, None) == _lib.TQD_ERR_BAD_ARG
    L.tqd_destroy(None)  # NULL-safe


def test_no_device_is_a_status_not_a_crash(L):
    torch = pytest.importorskip("torch")
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    m = synth.make_model(synth.TINY, 0)
    with pytest.raises(tqd.TQDError) as ei:
        tqd.Decoder(m, 16)
    assert ei.value.name == "TQD_ERR_NO_DEVICE"
    with pytest.raises(tqd.TQDError) as ei:
        tqd.Decoder.synthetic(synth.TINY, 0, 16)
    assert ei.value.name == "TQD_ERR_NO_DEVICE"


def test_scratch_size_queries(L):
    assert L.tqd_attention_scratch_bytes(16, 8, 128, 19) == 4 * (16 * 19 * 128 + 16 * 19 * 2 + 8)
    assert L.tqd_attention_scratch_bytes(0, 8, 128, 19) == 0
    assert L.tqd_argmax_scratch_bytes() > 0


def _c_layout(struct: str, fields):
    """sizeof and offsetof of a header struct, from a C program that
    includes include/tqd.h (compiled with gcc)."""
    import shutil
    import subprocess
    import tempfile
    cc = shutil.which("gcc") or shutil.which("cc")
    if not cc:
        pytest.skip("no C compiler")
    body = "\n".join(f'  printf("%zu\\n", offsetof({struct}, {f}));' for f in fields)
    src = ("#include <stddef.h>\n#include <stdio.h>\n#include \"tqd.h\"\n"
           f"int main(void) {{\n  printf(\"%zu\\n\", sizeof({struct}));\n{body}\n  return 0;\n}}\n")
    with tempfile.TemporaryDirectory() as d:
        c, exe = os.path.join(d, "layout.c"), os.path.join(d, "layout")
        open(c, "w").write(src)
        subprocess.run([cc, "-I", os.path.dirname(HEADER), c, "-o", exe], check=True, capture_output=True)
        out = subprocess.run([exe], check=True, capture_output=True, text=True).stdout.split()
    return int(out[0]), [int(x) for x in out[1:]]


@pytest.mark.parametrize("name, cls", [("tqd_config", _lib.tqd_config), ("tqd_sampling", _lib.tqd_sampling),
                                       ("tqd_layer_weights", _lib.tqd_layer_weights),
                                       ("tqd_host_weights", _lib.tqd_host_weights)])
def test_binding_structs_match_the_header_layout(name, cls):
    fields = [f[0] for f in cls._fields_]
    size, offsets = _c_layout(name, fields)
    assert ctypes.sizeof(cls) == size, name
    assert [getattr(cls, f).offset for f in fields] == offsets, name


def _build_client(d):
    """tests/c/tqd_client.c compiled against include/tqd.h and linked to the
    in-tree libtqd.so (rpath to its directory)."""
    import shutil
    import subprocess
    cc = shutil.which("gcc") or shutil.which("cc")
    if not cc:
        pytest.skip("no C compiler")
    lib = _lib.LIB_PATH
    if not os.path.exists(lib):
        pytest.skip("libtqd is not built")
    src = os.path.join(os.path.dirname(os.path.abspath(__file__)), "c", "tqd_client.c")
    exe = os.path.join(d, "tqd_client")
    libdir = os.path.dirname(lib)
    subprocess.run([cc, "-std=c11", "-Wall", "-Werror", "-I", os.path.dirname(HEADER), src, "-o", exe,
                    "-L", libdir, "-ltqd", f"-Wl,-rpath,{libdir}"], check=True, capture_output=True)
    return exe


def test_c_client_compiles_and_links_against_the_library():
    """A C program that uses only include/tqd.h and libtqd.so builds (its run
    is a GPU test: tests/test_gpu_synthetic.py)."""
    import tempfile
    with tempfile.TemporaryDirectory() as d:
        exe = _build_client(d)
        assert os.path.exists(exe)
