"""Plain CPU oracle of one batch-1 Llama-style decode step (ctypes wrapper).

TEST INFRASTRUCTURE. Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import this package. The product path
(``decode_megakernel_persistent_gb300``) never imports it, and the two share no
code: the arithmetic lives in ``oracle.c``, compiled here with gcc into
``liboracle.so`` in a float (``orc32_``) and a double (``orc64_``) flavour.

What the oracle computes, and which passage of the page "Hazy Research
Llama-3.2-1B Megakernel" each step follows, is written at the top of
``oracle.c``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_SRC = os.path.join(_HERE, "oracle.c")
_HDR = os.path.join(_HERE, "oracle.h")
_lib = None


def build(force: bool = False) -> str:
    """Compile oracle.c twice (float and double) into liboracle.so with gcc.

    -ffp-contract=off keeps gcc from fusing a*b+c into an FMA, so x86 and Arm
    builds round the same way.
    """
    newest_src = max(os.path.getmtime(_SRC), os.path.getmtime(_HDR))
    if not force and os.path.exists(_LIB_PATH) and os.path.getmtime(_LIB_PATH) >= newest_src:
        return _LIB_PATH
    bdir = os.path.join(_HERE, "_build")
    os.makedirs(bdir, exist_ok=True)
    common = ["gcc", "-O2", "-fPIC", "-fopenmp", "-ffp-contract=off", "-std=c11", "-Wall"]
    objs = []
    for real, prefix, is_double in (("float", "orc32_", 0), ("double", "orc64_", 1)):
        obj = os.path.join(bdir, f"oracle_{prefix}.o")
        subprocess.check_call(common + [
            f"-DORC_REAL={real}", f"-DORC_PREFIX={prefix}", f"-DORC_IS_DOUBLE={is_double}",
            "-c", _SRC, "-o", obj])
        objs.append(obj)
    tmp = _LIB_PATH + ".tmp"
    subprocess.check_call(["gcc", "-shared", "-fopenmp", *objs, "-o", tmp, "-lm"])
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


class _Config(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int) for n in (
        "n_layers", "hidden", "n_q_heads", "n_kv_heads", "head_dim", "inter", "vocab",
        "max_seq", "tied")] + [("rms_eps", ctypes.c_double), ("rope_theta", ctypes.c_double)]


_P16 = ctypes.POINTER(ctypes.c_uint16)
_PP16 = ctypes.POINTER(_P16)


class _Weights(ctypes.Structure):
    _fields_ = [("embed", _P16), ("lm_head", _P16), ("final_norm", _P16)] + [
        (n, _PP16) for n in ("attn_norm", "wq", "wk", "wv", "wo", "mlp_norm", "wg", "wu", "wd")]


def _load():
    global _lib
    if _lib is not None:
        return _lib
    build()
    lib = ctypes.CDLL(_LIB_PATH)
    for p, real in (("orc32_", ctypes.c_float), ("orc64_", ctypes.c_double)):
        preal = ctypes.POINTER(real)
        sig = {
            "to_bf16": (ctypes.c_uint16, [real]),
            "from_bf16": (real, [ctypes.c_uint16]),
            "rmsnorm": (None, [preal, _P16, ctypes.c_int, ctypes.c_double, preal]),
            "matvec": (None, [_P16, preal, ctypes.c_int, ctypes.c_int, preal]),
            "rope": (None, [preal, ctypes.c_int, ctypes.c_int, ctypes.c_double]),
            "silu": (real, [real]),
            "attention": (None, [preal, _P16, _P16, ctypes.c_int, ctypes.c_int, preal]),
            "argmax": (ctypes.c_int, [preal, ctypes.c_int]),
            "decode_step": (ctypes.c_int, [ctypes.POINTER(_Config), ctypes.POINTER(_Weights),
                                           _P16, _P16, ctypes.c_int, ctypes.c_int, preal]),
        }
        for name, (res, args) in sig.items():
            fn = getattr(lib, p + name)
            fn.restype = res
            fn.argtypes = args
    lib.orc_num_threads.restype = ctypes.c_int
    lib.orc_num_threads.argtypes = []
    lib.orc_set_threads.restype = None
    lib.orc_set_threads.argtypes = [ctypes.c_int]
    _lib = lib
    return lib


def _dtype(prec: int):
    if prec not in (32, 64):
        raise ValueError("prec must be 32 or 64")
    return np.float32 if prec == 32 else np.float64


def _fn(prec: int, name: str):
    return getattr(_load(), ("orc32_" if prec == 32 else "orc64_") + name)


def _preal(a: np.ndarray, prec: int):
    assert a.dtype == _dtype(prec) and a.flags.c_contiguous
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_float if prec == 32 else ctypes.c_double))


def _p16(a: np.ndarray):
    assert a.dtype == np.uint16 and a.flags.c_contiguous
    return a.ctypes.data_as(_P16)


def num_threads() -> int:
    """Threads the oracle's row-parallel matrix-vector products use."""
    return int(_load().orc_num_threads())


def set_threads(n: int) -> None:
    """Threads for the row-parallel loops from now on (timing only: each output
    row is summed by one thread, so results do not depend on it)."""
    _load().orc_set_threads(int(n))


# ---- primitives (used by the pin tests) -------------------------------------

def to_bf16(values, prec: int = 32) -> np.ndarray:
    fn = _fn(prec, "to_bf16")
    flat = np.asarray(values, dtype=_dtype(prec)).ravel()
    return np.array([fn(float(v)) for v in flat], dtype=np.uint16).reshape(np.shape(values))


def from_bf16(bits, prec: int = 32) -> np.ndarray:
    fn = _fn(prec, "from_bf16")
    flat = np.asarray(bits, dtype=np.uint16).ravel()
    return np.array([fn(int(b)) for b in flat], dtype=_dtype(prec)).reshape(np.shape(bits))


def rmsnorm(x, g_bits, eps: float, prec: int = 32) -> np.ndarray:
    x = np.ascontiguousarray(x, dtype=_dtype(prec))
    g = np.ascontiguousarray(g_bits, dtype=np.uint16)
    out = np.empty_like(x)
    _fn(prec, "rmsnorm")(_preal(x, prec), _p16(g), x.size, eps, _preal(out, prec))
    return out


def matvec(w_bits, x, prec: int = 32) -> np.ndarray:
    w = np.ascontiguousarray(w_bits, dtype=np.uint16)
    x = np.ascontiguousarray(x, dtype=_dtype(prec))
    rows, cols = w.shape
    assert x.size == cols
    y = np.empty(rows, dtype=_dtype(prec))
    _fn(prec, "matvec")(_p16(w), _preal(x, prec), rows, cols, _preal(y, prec))
    return y


def rope(v, pos: int, theta: float, prec: int = 32) -> np.ndarray:
    out = np.array(v, dtype=_dtype(prec), copy=True)
    _fn(prec, "rope")(_preal(out, prec), out.size, pos, theta)
    return out


def silu(z: float, prec: int = 32) -> float:
    return float(_fn(prec, "silu")(z))


def attention(q, k_bits, v_bits, prec: int = 32) -> np.ndarray:
    q = np.ascontiguousarray(q, dtype=_dtype(prec))
    k = np.ascontiguousarray(k_bits, dtype=np.uint16)
    v = np.ascontiguousarray(v_bits, dtype=np.uint16)
    n_pos, hd = k.shape
    assert q.size == hd and v.shape == k.shape
    out = np.empty(hd, dtype=_dtype(prec))
    _fn(prec, "attention")(_preal(q, prec), _p16(k), _p16(v), n_pos, hd, _preal(out, prec))
    return out


def argmax(v, prec: int = 32) -> int:
    v = np.ascontiguousarray(v, dtype=_dtype(prec))
    return int(_fn(prec, "argmax")(_preal(v, prec), v.size))


# ---- whole decode step --------------------------------------------------------

class OracleModel:
    """A model held in host memory (bf16 bit patterns) plus the oracle's own KV cache.

    ``weights`` maps names to uint16 numpy arrays: ``embed`` [V,H], ``final_norm`` [H],
    optional ``lm_head`` [V,H], and per-layer lists ``attn_norm``, ``wq``, ``wk``,
    ``wv``, ``wo``, ``mlp_norm``, ``wg``, ``wu``, ``wd``.
    """

    LAYER_KEYS = ("attn_norm", "wq", "wk", "wv", "wo", "mlp_norm", "wg", "wu", "wd")

    def __init__(self, cfg: dict, weights: dict, max_seq: int, prec: int = 32):
        self.prec = prec
        self.cfg = dict(cfg)
        self.max_seq = max_seq
        c = _Config()
        for n in ("n_layers", "hidden", "n_q_heads", "n_kv_heads", "head_dim", "inter",
                  "vocab"):
            setattr(c, n, int(cfg[n]))
        c.max_seq = int(max_seq)
        c.tied = int(bool(cfg["tied"]))
        c.rms_eps = float(cfg["rms_eps"])
        c.rope_theta = float(cfg["rope_theta"])
        self._c = c
        self._keep = []

        def arr(a):
            a = np.ascontiguousarray(a, dtype=np.uint16)
            self._keep.append(a)
            return a

        w = _Weights()
        w.embed = _p16(arr(weights["embed"]))
        w.final_norm = _p16(arr(weights["final_norm"]))
        w.lm_head = _p16(arr(weights["lm_head"])) if not cfg["tied"] else _P16()
        L = int(cfg["n_layers"])
        for key in self.LAYER_KEYS:
            ptrs = (_P16 * max(L, 1))()
            for i in range(L):
                ptrs[i] = _p16(arr(weights[key][i]))
            self._keep.append(ptrs)
            setattr(w, key, ctypes.cast(ptrs, _PP16))
        self._w = w
        shape = (L, int(cfg["n_kv_heads"]), int(max_seq), int(cfg["head_dim"]))
        self.k_cache = np.zeros(shape, dtype=np.uint16)
        self.v_cache = np.zeros(shape, dtype=np.uint16)

    def decode_step(self, token: int, pos: int):
        """Run one step; returns (logits, next_token). Writes k, v at ``pos``."""
        logits = np.empty(int(self.cfg["vocab"]), dtype=_dtype(self.prec))
        nxt = _fn(self.prec, "decode_step")(
            ctypes.byref(self._c), ctypes.byref(self._w), _p16(self.k_cache),
            _p16(self.v_cache), int(token), int(pos), _preal(logits, self.prec))
        if nxt < 0:
            raise ValueError(f"oracle decode_step rejected token={token} pos={pos} ({nxt})")
        return logits, int(nxt)
