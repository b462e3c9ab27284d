"""The C ABI without a GPU: the library loads, exports every function that
include/ll.h declares, its structures have the layout the binding assumes, its
constants match, and argument and shape checks answer before any device work."""
import ctypes
import os
import re
import subprocess

import pytest

from decode_megakernel_persistent_gb300 import build as llbuild
from decode_megakernel_persistent_gb300 import ll

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "ll.h")


@pytest.fixture(scope="module")
def lib():
    llbuild.build()
    return ll.lib()


def header_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(ll_[a-z_]+)\s*\(", text)))


def test_exports_every_declared_function(lib):
    declared = header_functions()
    assert set(declared) == set(ll.EXPORTS)
    out = subprocess.run(["nm", "-D", "--defined-only", ll.LIB_PATH], capture_output=True, text=True).stdout
    exported = set(re.findall(r" T (ll_[a-z_]+)$", out, flags=re.M))
    for name in declared:
        assert name in exported, name
        assert hasattr(lib, name)


def test_constants_match_header():
    text = open(HEADER).read()
    for name, val in re.findall(r"#define (LL_[A-Z0-9_]+) \(?(-?\d+)\)?", text):
        assert getattr(ll, name) == int(val), name


def test_struct_layout_matches_c(tmp_path):
    src = tmp_path / "layout.c"
    src.write_text(r'''
#include <stdio.h>
#include <stddef.h>
#include "ll.h"
int main(void) {
  printf("%zu %zu %zu %zu %zu\n", sizeof(ll_config), offsetof(ll_config, rms_eps),
         offsetof(ll_config, rope_theta), sizeof(ll_weights), offsetof(ll_weights, wd));
  return 0;
}
''')
    exe = tmp_path / "layout"
    subprocess.check_call(["gcc", "-I", os.path.join(ROOT, "include"), str(src), "-o", str(exe)])
    got = [int(v) for v in subprocess.check_output([str(exe)]).split()]
    want = [ctypes.sizeof(ll.ll_config), ll.ll_config.rms_eps.offset, ll.ll_config.rope_theta.offset,
            ctypes.sizeof(ll.ll_weights), ll.ll_weights.wd.offset]
    assert got == want


def _init(lib, cfg, weights=None, k=16, v=16):
    h = ctypes.c_void_p()
    w = weights if weights is not None else ll.ll_weights()
    rc = lib.ll_init(ctypes.byref(cfg) if cfg is not None else None, ctypes.byref(w), k, v, None,
                     ctypes.byref(h))
    return rc, h, lib.ll_init_error().decode()


def good_config():
    c = ll.ll_config()
    c.n_layers, c.hidden, c.n_q_heads, c.n_kv_heads, c.head_dim = 2, 256, 4, 2, 64
    c.inter, c.vocab, c.max_seq, c.tied, c.backend = 1024, 4096, 64, 1, 0
    c.rms_eps, c.rope_theta = 1e-5, 500000.0
    return c


def test_init_rejects_null_and_bad_shapes(lib):
    rc, h, msg = _init(lib, None)
    assert rc == ll.LL_ERR_ARG and not h.value
    for field, value in (("head_dim", 96), ("hidden", 200), ("inter", 1000), ("n_kv_heads", 3),
                         ("n_layers", 0), ("max_seq", 0)):
        c = good_config()
        setattr(c, field, value)
        rc, h, msg = _init(lib, c)
        assert rc == ll.LL_ERR_SHAPE, (field, rc, msg)
        assert not h.value and msg
    c = good_config()
    c.n_q_heads, c.n_kv_heads = 32, 2  # 16 query heads per KV head
    assert _init(lib, c)[0] == ll.LL_ERR_SHAPE
    c = good_config()
    c.backend = 7
    assert _init(lib, c)[0] == ll.LL_ERR_ARG


def test_init_rejects_misaligned_or_missing_pointers(lib):
    c = good_config()
    rc, _, msg = _init(lib, c, k=18, v=32)  # misaligned K cache
    assert rc == ll.LL_ERR_ARG and "aligned" in msg
    w = ll.ll_weights()
    w.embed, w.final_norm = 4096, 8192
    rc, _, msg = _init(lib, c, weights=w, k=32, v=48)  # per-layer arrays missing
    assert rc == ll.LL_ERR_ARG and "NULL" in msg
    arrs = []
    for key in ll.LAYER_KEYS:
        a = (ctypes.c_void_p * 2)(4096 * 3, 4096 * 5 + (2 if key == "wd" else 0))
        arrs.append(a)
        setattr(w, key, ctypes.cast(a, ctypes.POINTER(ctypes.c_void_p)))
    rc, _, msg = _init(lib, c, weights=w, k=32, v=48)
    assert rc == ll.LL_ERR_ARG and "layer 1" in msg


def test_null_handle_calls_are_safe(lib):
    assert lib.ll_decode_step(None, 0, 0, None, None) == ll.LL_ERR_ARG
    assert lib.ll_decode_step_async(None, None, 0, None, None) == ll.LL_ERR_ARG
    assert lib.ll_synchronize(None) == ll.LL_ERR_ARG
    assert lib.ll_set_timeout_ns(None, 5) == ll.LL_ERR_ARG
    v = ctypes.c_int64()
    assert lib.ll_query(None, 0, ctypes.byref(v)) == ll.LL_ERR_ARG
    assert lib.ll_debug_inject(None, 0, 0, 0) == ll.LL_ERR_ARG
    assert lib.ll_last_error(None) == b"null handle"
    lib.ll_free(None)
