"""Thin ctypes binding of libll.so (the C ABI in include/ll.h).

Every function here has the name of the C entry point it calls and does only
argument marshalling: torch tensors supply device pointers and the stream, and
every step of the decode runs in the library's CUDA kernels. There is no
fallback: if libll.so is missing or fails to load, the first call raises.
"""
from __future__ import annotations

import ctypes
import os

LL_OK = 0
LL_ERR_ARG = -1
LL_ERR_SHAPE = -2
LL_ERR_CUDA = -3
LL_ERR_DEP_TIMEOUT = -4
LL_ERR_OOM = -5
LL_ERR_DEVICE = -6
LL_ERR_NUMERIC = -7

LL_BACKEND_MEGAKERNEL = 0
LL_BACKEND_CHAIN = 1

LL_Q_NUM_SMS = 0
LL_Q_ATTN_SPLITS = 1
LL_Q_PAGE_BYTES = 2
LL_Q_NUM_PAGES = 3
LL_Q_SCRATCH_BYTES = 4
LL_Q_MAX_INSTRS = 5
LL_Q_LAUNCHES_PER_STEP = 6
LL_Q_SMEM_BYTES = 7
LL_Q_TRACE_BYTES = 8
LL_Q_MV_TC = 9
LL_Q_BATCH_CC = 12
LL_Q_BATCH = 10
LL_MAX_BATCH = 8

LL_STATIC_SCRATCH_BYTES = 4194304
LL_STATIC_MAX_LAYERS = 256

LL_FAULT_NONE = 0
LL_FAULT_DROP_SIGNAL = 1

OP_QKV, OP_ATTN, OP_OPROJ, OP_GATEUP, OP_DOWN = range(5)

LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libll.so")

EXPORTS = ("ll_init", "ll_init_error", "ll_decode_step", "ll_decode_step_async", "ll_decode_steps", "ll_synchronize",
           "ll_set_trace", "ll_set_timeout_ns", "ll_query", "ll_debug_inject", "ll_plan", "ll_last_error",
           "ll_free", "ll_decode_step_static", "ll_init_batch", "ll_decode_steps_batch", "ll_handle_plan",
           "ll_prefill")


class LLError(RuntimeError):
    def __init__(self, code: int, msg: str):
        super().__init__(f"libll error {code}: {msg}")
        self.code = code


class ll_config(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in (
        "n_layers", "hidden", "n_q_heads", "n_kv_heads", "head_dim", "inter", "vocab", "max_seq",
        "tied", "backend")] + [("rms_eps", ctypes.c_float), ("rope_theta", ctypes.c_float)]


_P16 = ctypes.c_void_p
_PP16 = ctypes.POINTER(ctypes.c_void_p)
LAYER_KEYS = ("attn_norm", "wq", "wk", "wv", "wo", "mlp_norm", "wg", "wu", "wd")


class ll_weights(ctypes.Structure):
    _fields_ = [("embed", _P16), ("lm_head", _P16), ("final_norm", _P16)] + [
        (k, _PP16) for k in LAYER_KEYS]


_lib = None


def lib() -> ctypes.CDLL:
    """Open libll.so (raises if it was not built)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise RuntimeError(f"{LIB_PATH} is missing: build it with __graft_entry__.build() "
                           "(there is no CPU fallback)")
    L = ctypes.CDLL(LIB_PATH)
    vp, i32, u64 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_uint64
    L.ll_init.argtypes = [ctypes.POINTER(ll_config), ctypes.POINTER(ll_weights), vp, vp, vp,
                          ctypes.POINTER(vp)]
    L.ll_init.restype = ctypes.c_int
    L.ll_init_error.argtypes = []
    L.ll_init_error.restype = ctypes.c_char_p
    L.ll_decode_step.argtypes = [vp, i32, i32, vp, ctypes.POINTER(i32)]
    L.ll_decode_step.restype = ctypes.c_int
    L.ll_decode_step_async.argtypes = [vp, vp, i32, vp, vp]
    L.ll_decode_step_async.restype = ctypes.c_int
    L.ll_decode_steps.argtypes = [vp, vp, i32, i32, vp, vp]
    L.ll_decode_steps.restype = ctypes.c_int
    L.ll_synchronize.argtypes = [vp]
    L.ll_synchronize.restype = ctypes.c_int
    L.ll_set_trace.argtypes = [vp, vp, ctypes.c_size_t]
    L.ll_set_trace.restype = ctypes.c_int
    L.ll_set_timeout_ns.argtypes = [vp, u64]
    L.ll_set_timeout_ns.restype = ctypes.c_int
    L.ll_query.argtypes = [vp, ctypes.c_int, ctypes.POINTER(ctypes.c_int64)]
    L.ll_query.restype = ctypes.c_int
    L.ll_debug_inject.argtypes = [vp, ctypes.c_int, ctypes.c_int, ctypes.c_int]
    L.ll_debug_inject.restype = ctypes.c_int
    L.ll_plan.argtypes = [ctypes.POINTER(ll_config), i32, vp, ctypes.c_size_t, ctypes.POINTER(i32)]
    L.ll_plan.restype = ctypes.c_int
    L.ll_last_error.argtypes = [vp]
    L.ll_last_error.restype = ctypes.c_char_p
    L.ll_free.argtypes = [vp]
    L.ll_free.restype = None
    L.ll_decode_step_static.argtypes = [ctypes.POINTER(ll_config), ctypes.POINTER(ll_weights), vp, vp, i32, i32,
                                        vp, ctypes.POINTER(i32), vp, ctypes.c_char_p, ctypes.c_size_t]
    L.ll_decode_step_static.restype = ctypes.c_int
    L.ll_init_batch.argtypes = [ctypes.POINTER(ll_config), ctypes.POINTER(ll_weights), ctypes.POINTER(vp),
                                ctypes.POINTER(vp), i32, vp, ctypes.POINTER(vp)]
    L.ll_init_batch.restype = ctypes.c_int
    L.ll_decode_steps_batch.argtypes = [vp, vp, ctypes.POINTER(i32), i32, vp, vp]
    L.ll_decode_steps_batch.restype = ctypes.c_int
    L.ll_handle_plan.argtypes = [vp, vp, ctypes.c_size_t, ctypes.POINTER(i32)]
    L.ll_handle_plan.restype = ctypes.c_int
    L.ll_prefill.argtypes = [vp, vp, i32, i32, vp, vp]
    L.ll_prefill.restype = ctypes.c_int
    _lib = L
    return L


def _ptr(t) -> int:
    return 0 if t is None else int(t.data_ptr())


def _check(h, rc: int):
    if rc != LL_OK:
        raise LLError(rc, lib().ll_last_error(h).decode())


def make_config(shape, max_seq: int, backend: int = LL_BACKEND_MEGAKERNEL) -> ll_config:
    """ll_config from a shape description with the attributes of synth.ModelShape."""
    c = ll_config()
    for n in ("n_layers", "hidden", "n_q_heads", "n_kv_heads", "head_dim", "inter", "vocab"):
        setattr(c, n, int(getattr(shape, n)))
    c.max_seq = int(max_seq)
    c.tied = int(bool(shape.tied))
    c.backend = int(backend)
    c.rms_eps = float(shape.rms_eps)
    c.rope_theta = float(shape.rope_theta)
    return c


def _weights_struct(weights: dict):
    """ll_weights for a dict of CUDA bf16 tensors, plus the host arrays it points into."""
    w = ll_weights()
    w.embed = _ptr(weights["embed"])
    w.final_norm = _ptr(weights["final_norm"])
    w.lm_head = _ptr(weights.get("lm_head"))
    keep = []
    for k in LAYER_KEYS:
        arr = (ctypes.c_void_p * max(1, len(weights[k])))(*[_ptr(t) for t in weights[k]])
        keep.append(arr)
        setattr(w, k, ctypes.cast(arr, _PP16))
    return w, keep


def ll_init(cfg: ll_config, weights: dict, k_cache, v_cache, stream=None):
    """Create a handle. ``weights`` maps names to CUDA bf16 tensors (per-layer names
    to lists); ``stream`` is a torch.cuda.Stream or None for torch's current stream."""
    import torch
    if stream is None:
        stream = torch.cuda.current_stream()
    w, keep = _weights_struct(weights)
    h = ctypes.c_void_p()
    rc = lib().ll_init(ctypes.byref(cfg), ctypes.byref(w), _ptr(k_cache), _ptr(v_cache),
                       ctypes.c_void_p(stream.cuda_stream), ctypes.byref(h))
    if rc != LL_OK:
        raise LLError(rc, lib().ll_init_error().decode())
    return h


def ll_decode_step(h, token: int, pos: int, logits=None) -> int:
    """Synchronous step; returns the greedy next token."""
    nxt = ctypes.c_int32(-1)
    _check(h, lib().ll_decode_step(h, int(token), int(pos), _ptr(logits), ctypes.byref(nxt)))
    return int(nxt.value)


def ll_decode_steps(h, token_dev, pos: int, n_steps: int, logits, tokens_dev) -> None:
    _check(h, lib().ll_decode_steps(h, _ptr(token_dev), int(pos), int(n_steps), _ptr(logits), _ptr(tokens_dev)))


def ll_decode_step_async(h, token_dev, pos: int, logits, next_token_dev) -> None:
    _check(h, lib().ll_decode_step_async(h, _ptr(token_dev), int(pos), _ptr(logits),
                                         _ptr(next_token_dev)))


def ll_synchronize(h) -> None:
    _check(h, lib().ll_synchronize(h))


def ll_set_trace(h, trace_dev=None) -> None:
    """Enable (a CUDA uint64/int64 tensor of LL_Q_TRACE_BYTES bytes) or disable (None) tracing."""
    nbytes = 0 if trace_dev is None else trace_dev.numel() * trace_dev.element_size()
    _check(h, lib().ll_set_trace(h, _ptr(trace_dev), nbytes))


def ll_set_timeout_ns(h, ns: int) -> None:
    _check(h, lib().ll_set_timeout_ns(h, int(ns)))


def ll_query(h, what: int) -> int:
    v = ctypes.c_int64()
    _check(h, lib().ll_query(h, int(what), ctypes.byref(v)))
    return int(v.value)


def ll_debug_inject(h, kind: int, layer: int = 0, op: int = 0) -> None:
    _check(h, lib().ll_debug_inject(h, int(kind), int(layer), int(op)))


def ll_plan(cfg: ll_config, nsm: int):
    """The schedule for `nsm` SMs as an int32 numpy array [nsm, max_instr, 7] (host only)."""
    import numpy as np
    mx = ctypes.c_int32()
    rc = lib().ll_plan(ctypes.byref(cfg), int(nsm), None, 0, ctypes.byref(mx))
    if rc != LL_OK:
        raise LLError(rc, "ll_plan rejected the configuration")
    out = np.zeros((int(nsm), mx.value, 7), dtype=np.int32)
    rc = lib().ll_plan(ctypes.byref(cfg), int(nsm), out.ctypes.data, out.size, ctypes.byref(mx))
    if rc != LL_OK:
        raise LLError(rc, "ll_plan failed")
    return out


def ll_prefill(h, tokens_dev, n: int, pos0: int, logits, next_token_dev) -> None:
    _check(h, lib().ll_prefill(h, _ptr(tokens_dev), int(n), int(pos0), _ptr(logits), _ptr(next_token_dev)))


def ll_handle_plan(h):
    """The handle's own schedule as an int32 numpy array [nsm, max_instr, 7]."""
    import numpy as np
    mx = ctypes.c_int32()
    _check(h, lib().ll_handle_plan(h, None, 0, ctypes.byref(mx)))
    nsm = ll_query(h, LL_Q_NUM_SMS)
    out = np.zeros((nsm, mx.value, 7), dtype=np.int32)
    _check(h, lib().ll_handle_plan(h, out.ctypes.data, out.size, ctypes.byref(mx)))
    return out


def ll_decode_step_static(cfg: ll_config, weights: dict, k_cache, v_cache, token: int, pos: int,
                          logits=None, stream=None) -> int:
    """One decode step without a handle and without device allocation; returns the
    greedy next token. ``stream`` is a torch.cuda.Stream or None for torch's current one."""
    import torch
    check_static_args(cfg, weights, k_cache, v_cache, logits)
    if stream is None:
        stream = torch.cuda.current_stream()
    w, keep = _weights_struct(weights)
    nxt = ctypes.c_int32(-1)
    err = ctypes.create_string_buffer(256)
    rc = lib().ll_decode_step_static(ctypes.byref(cfg), ctypes.byref(w), _ptr(k_cache), _ptr(v_cache), int(token),
                                     int(pos), _ptr(logits), ctypes.byref(nxt), ctypes.c_void_p(stream.cuda_stream),
                                     err, len(err))
    del keep
    if rc != LL_OK:
        raise LLError(rc, err.value.decode())
    return int(nxt.value)


def ll_init_batch(cfg: ll_config, weights: dict, k_caches, v_caches, stream=None):
    """A batched handle: one (k, v) cache pair per sequence (lists of CUDA bf16 tensors)."""
    import torch
    if stream is None:
        stream = torch.cuda.current_stream()
    w, keep = _weights_struct(weights)
    n = len(k_caches)
    kp = (ctypes.c_void_p * max(1, n))(*[_ptr(t) for t in k_caches])
    vp_ = (ctypes.c_void_p * max(1, len(v_caches)))(*[_ptr(t) for t in v_caches])
    h = ctypes.c_void_p()
    rc = lib().ll_init_batch(ctypes.byref(cfg), ctypes.byref(w), kp, vp_, int(n), ctypes.c_void_p(stream.cuda_stream),
                             ctypes.byref(h))
    if rc != LL_OK:
        raise LLError(rc, lib().ll_init_error().decode())
    return h


def ll_decode_steps_batch(h, tokens_in_dev, positions, n_steps: int, logits, tokens_dev) -> None:
    pos = (ctypes.c_int32 * max(1, len(positions)))(*[int(x) for x in positions])
    _check(h, lib().ll_decode_steps_batch(h, _ptr(tokens_in_dev), pos, int(n_steps), _ptr(logits), _ptr(tokens_dev)))


def ll_last_error(h) -> str:
    return lib().ll_last_error(h).decode()


def ll_free(h) -> None:
    if h:
        lib().ll_free(h)


def _need(t, name: str, dtype, min_numel: int, device, optional: bool = True) -> None:
    """The library takes raw device pointers and cannot see a buffer's size, so
    the buffers a step writes or reads are checked here: a CUDA tensor of the
    right dtype on the decoder's device, contiguous, with room for min_numel
    elements (raises LLError(LL_ERR_ARG) before anything is launched)."""
    if t is None:
        if optional:
            return
        raise LLError(LL_ERR_ARG, f"{name} is required")
    if not getattr(t, "is_cuda", False):
        raise LLError(LL_ERR_ARG, f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise LLError(LL_ERR_ARG, f"{name} must be {dtype}, not {t.dtype}")
    if device is not None and t.device != device:
        raise LLError(LL_ERR_ARG, f"{name} is on {t.device}, the decoder on {device}")
    if not t.is_contiguous():
        raise LLError(LL_ERR_ARG, f"{name} must be contiguous")
    if t.numel() < min_numel:
        raise LLError(LL_ERR_ARG, f"{name} holds {t.numel()} elements, the call needs {min_numel}")


def check_model(shape, weights: dict, k_cache, v_cache, max_seq: int) -> None:
    """The weights and caches ll_init will read, against the shape: every tensor a
    contiguous CUDA bf16 tensor on the embedding's device with exactly the
    elements of its matrix or vector (per-layer lists n_layers long), and the
    caches room for [n_layers][n_kv_heads][max_seq][head_dim] (raises
    LLError(LL_ERR_ARG) naming the first misfit)."""
    import torch
    H, V, I, L = int(shape.hidden), int(shape.vocab), int(shape.inter), int(shape.n_layers)
    q, kv = int(shape.n_q_heads) * int(shape.head_dim), int(shape.n_kv_heads) * int(shape.head_dim)
    dev = getattr(weights.get("embed"), "device", None)

    def exact(t, name, n):
        _need(t, name, torch.bfloat16, n, dev, optional=False)
        if t.numel() != n:
            raise LLError(LL_ERR_ARG, f"{name} holds {t.numel()} elements, the shape has {n}")

    exact(weights.get("embed"), "embed", V * H)
    exact(weights.get("final_norm"), "final_norm", H)
    if not shape.tied:
        exact(weights.get("lm_head"), "lm_head", V * H)
    per_layer = {"attn_norm": H, "wq": q * H, "wk": kv * H, "wv": kv * H, "wo": H * q,
                 "mlp_norm": H, "wg": I * H, "wu": I * H, "wd": H * I}
    for key, n in per_layer.items():
        ts = weights.get(key)
        if ts is None or len(ts) != L:
            raise LLError(LL_ERR_ARG, f"{key} must list one tensor per layer ({L})")
        for i, t in enumerate(ts):
            exact(t, f"{key}[{i}]", n)
    cache = L * kv * int(max_seq)
    _need(k_cache, "k_cache", torch.bfloat16, cache, dev, optional=False)
    _need(v_cache, "v_cache", torch.bfloat16, cache, dev, optional=False)


def check_static_args(cfg: ll_config, weights: dict, k_cache, v_cache, logits) -> None:
    """What ll_decode_step_static will read and write, against cfg: one tensor per
    layer in every per-layer list (the C side walks n_layers entries of each),
    every weight of its exact size, caches with room for
    [n_layers][n_kv_heads][max_seq][head_dim], logits (if given) with room for
    vocab floats, all on one device, and that device torch's current one, which
    the library sets up from cudaGetDevice (raises LLError(LL_ERR_ARG))."""
    import types

    import torch
    L = int(cfg.n_layers)
    for key in LAYER_KEYS:
        ts = weights.get(key)
        if ts is None or len(ts) != L:
            raise LLError(LL_ERR_ARG, f"{key} must list one tensor per layer ({L})")
    shape = types.SimpleNamespace(**{n: int(getattr(cfg, n)) for n in (
        "n_layers", "hidden", "n_q_heads", "n_kv_heads", "head_dim", "inter", "vocab")}, tied=bool(cfg.tied))
    check_model(shape, weights, k_cache, v_cache, int(cfg.max_seq))
    dev = weights["embed"].device
    _need(logits, "logits", torch.float32, int(cfg.vocab), dev)
    cur = torch.device("cuda", torch.cuda.current_device())
    if dev != cur:
        raise LLError(LL_ERR_ARG, f"the tensors are on {dev}, torch's current device is {cur}")


class Decoder:
    """Owns a handle plus references to the tensors it points into. The model's
    tensors are checked at construction (check_model) and the buffers of every
    step before its library call (_need)."""

    def __init__(self, shape, weights: dict, k_cache, v_cache, max_seq: int,
                 backend: int = LL_BACKEND_MEGAKERNEL, stream=None):
        import torch
        self.handle = None
        check_model(shape, weights, k_cache, v_cache, max_seq)
        self.shape = shape
        self.weights = weights
        self.k_cache, self.v_cache = k_cache, v_cache
        self.stream = stream if stream is not None else torch.cuda.current_stream()
        self.cfg = make_config(shape, max_seq, backend)
        self.device = getattr(weights["embed"], "device", None)
        self.handle = ll_init(self.cfg, weights, k_cache, v_cache, self.stream)

    def _bufs(self, token_dev, logits, n_logits: int, out, n_out: int, out_required: bool = False) -> None:
        import torch
        V = int(self.shape.vocab)
        if token_dev is not None:
            _need(token_dev, "token_dev", torch.int32, 1, self.device, optional=False)
        _need(logits, "logits", torch.float32, n_logits * V, self.device)
        _need(out, "next-token buffer", torch.int32, n_out, self.device, optional=not out_required)

    def step(self, token: int, pos: int, logits=None) -> int:
        self._bufs(None, logits, 1, None, 0)
        return ll_decode_step(self.handle, token, pos, logits)

    def step_async(self, token_dev, pos: int, logits, next_token_dev) -> None:
        self._bufs(token_dev, logits, 1, next_token_dev, 1)
        ll_decode_step_async(self.handle, token_dev, pos, logits, next_token_dev)

    def steps(self, token_dev, pos: int, n_steps: int, logits, tokens_dev) -> None:
        n = max(int(n_steps), 0)
        self._bufs(token_dev, logits, n, tokens_dev, n, out_required=True)
        ll_decode_steps(self.handle, token_dev, pos, n_steps, logits, tokens_dev)

    def prefill(self, tokens_dev, pos0: int, logits, next_token_dev) -> None:
        """All of tokens_dev (int32 [n]) at positions pos0..pos0+n-1 in one pass;
        the last position's logits ([vocab] fp32, or None) and greedy token."""
        import torch
        n = int(tokens_dev.numel()) if tokens_dev is not None else 0
        _need(tokens_dev, "tokens_dev", torch.int32, max(n, 1), self.device, optional=False)
        _need(logits, "logits", torch.float32, int(self.shape.vocab), self.device)
        _need(next_token_dev, "next_token_dev", torch.int32, 1, self.device, optional=False)
        ll_prefill(self.handle, tokens_dev, n, pos0, logits, next_token_dev)

    def synchronize(self) -> None:
        ll_synchronize(self.handle)

    def query(self, what: int) -> int:
        return ll_query(self.handle, what)

    def close(self) -> None:
        if self.handle:
            ll_free(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


class BatchDecoder(Decoder):
    """A batched handle (ll_init_batch) plus references to the tensors it points
    into: n sequences, one (k, v) cache pair each, share every pass over the
    weights. The model's tensors and every cache are checked at construction, the
    buffers of every launch before its library call."""

    def __init__(self, shape, weights: dict, k_caches, v_caches, max_seq: int, stream=None):
        import torch
        self.handle = None
        n = len(k_caches)
        if n not in (1, 2, 4, 8) or len(v_caches) != n:
            raise LLError(LL_ERR_ARG, "the batch must be 1, 2, 4 or 8 sequences, one (k, v) cache pair each")
        for k, v in zip(k_caches, v_caches):
            check_model(shape, weights, k, v, max_seq)
        self.n = n
        self.shape = shape
        self.weights = weights
        self.k_caches, self.v_caches = list(k_caches), list(v_caches)
        self.stream = stream if stream is not None else torch.cuda.current_stream()
        self.cfg = make_config(shape, max_seq, LL_BACKEND_MEGAKERNEL)
        self.device = getattr(weights["embed"], "device", None)
        self.handle = ll_init_batch(self.cfg, weights, self.k_caches, self.v_caches, self.stream)

    def steps_batch(self, tokens_in_dev, positions, n_steps: int, logits, tokens_dev) -> None:
        """n_steps greedy steps of every sequence in one launch: tokens_in_dev [n]
        int32, positions a host list of n first positions, logits [n_steps][n][vocab]
        fp32 or None, tokens_dev [n_steps][n] int32."""
        import torch
        if len(positions) != self.n:
            raise LLError(LL_ERR_ARG, f"{self.n} positions needed, got {len(positions)}")
        steps = max(int(n_steps), 0)
        _need(tokens_in_dev, "tokens_in_dev", torch.int32, self.n, self.device, optional=False)
        _need(logits, "logits", torch.float32, steps * self.n * int(self.shape.vocab), self.device)
        _need(tokens_dev, "tokens_dev", torch.int32, steps * self.n, self.device, optional=False)
        ll_decode_steps_batch(self.handle, tokens_in_dev, positions, n_steps, logits, tokens_dev)
