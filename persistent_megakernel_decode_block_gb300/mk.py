"""Thin ctypes binding of libmk.so (include/mk.h): argument marshalling only.

Every function keeps the C name and returns what the C call returns or raises
MkError on a non-zero code.  Tensors may be torch tensors (their data_ptr()),
numpy arrays (host memory) or raw integer addresses.  There is no fallback:
if libmk.so is missing the import fails loudly; build it with
`python -c "import __graft_entry__ as g; g.build()"`.
"""
import ctypes
import os

import numpy as np

from ._build import LIB

MK_OK = 0
ERRORS = {-1: "MK_ERR_CONFIG", -2: "MK_ERR_ARG", -3: "MK_ERR_DEVICE", -4: "MK_ERR_NOMEM",
          -5: "MK_ERR_STATE", -6: "MK_ERR_TIMEOUT", -7: "MK_ERR_BOUNDS", -8: "MK_ERR_LAUNCH",
          -9: "MK_ERR_CUDA"}
for _c, _n in ERRORS.items():
    globals()[_n] = _c
MK_OP_QKV, MK_OP_ATTN, MK_OP_OPROJ, MK_OP_GATEUP, MK_OP_DOWN, MK_OP_LMHEAD = 1, 2, 3, 4, 5, 6
MK_NO_COUNTER = 0xFFFFFFFF
MK_FLAG_TRACE, MK_FLAG_HOST_ONLY, MK_FLAG_FAULT_WAIT, MK_FLAG_STREAM_B1 = 1, 2, 4, 8
MK_FLAG_FP8_WEIGHTS = 0x10
MK_SCHED_DYNAMIC, MK_SCHED_STATIC, MK_SCHED_HYBRID = 0, 1, 2
MK_LIST_ATTN = 0x80000000  # hybrid lists: entry MK_LIST_ATTN | l = layer l's attention queue

_i32, _u32, _f32, _vp = ctypes.c_int32, ctypes.c_uint32, ctypes.c_float, ctypes.c_void_p


class mk_config(ctypes.Structure):
    _fields_ = [(n, _i32) for n in ("n_layers", "hidden", "n_q_heads", "n_kv_heads", "head_dim",
                                    "ffn_dim", "vocab")] + [
        ("rms_eps", _f32), ("rope_theta", _f32), ("tie_embeddings", _i32), ("batch", _i32),
        ("max_ctx", _i32), ("sched_mode", _i32), ("flags", _u32), ("wait_timeout_us", _i32),
        ("num_sms", _i32), ("smem_bytes", _i32), ("page_bytes", _i32), ("attn_chunk", _i32),
        ("l2_prefetch_kb", _i32)]


class mk_plan_info_t(ctypes.Structure):
    _fields_ = [(n, _u32) for n in ("n_instr", "n_counters", "n_wait_counters", "n_phases",
                                    "n_blocks", "threads", "ring_pages", "page_bytes",
                                    "fifo_depth", "smem_bytes", "attn_nchunk", "attn_chunk")] + [
        ("arena_bytes", ctypes.c_uint64), ("weight_bytes", ctypes.c_uint64),
        ("warp_ring_slots", _u32), ("kernel", _u32)]


class mk_phase(ctypes.Structure):
    _fields_ = [(n, _u32) for n in ("first", "count", "op", "layer")]


LAYER_FIELDS = ("attn_norm", "wq", "wk", "wv", "wo", "mlp_norm", "w_gate", "w_up", "w_down")


class mk_layer_weights(ctypes.Structure):
    _fields_ = [(n, _vp) for n in LAYER_FIELDS]


class mk_weights(ctypes.Structure):
    _fields_ = [("embed", _vp), ("final_norm", _vp), ("lm_head", _vp),
                ("layers", ctypes.POINTER(mk_layer_weights))]


class mk_kv_cache(ctypes.Structure):
    _fields_ = [("k", _vp), ("v", _vp)]


class mk_debug_buffers_t(ctypes.Structure):
    _fields_ = [(n, _vp) for n in ("x", "q", "attn", "h")]


# numpy view of the 64-byte instruction record (layout of mk_instr in mk.h)
INSTR_DTYPE = np.dtype([("op", "u1"), ("flags", "u1"), ("layer", "<u2"), ("b", "<u2"),
                        ("g", "<u2"), ("wait_ctr", "<u4"), ("wait_tgt", "<u4"),
                        ("sig_ctr", "<u4"), ("sig2_ctr", "<u4"), ("sig2_after", "<u4"),
                        ("row0", "<u4"), ("nrows", "<u4"), ("chunk", "<u4"), ("nchunk", "<u4"),
                        ("npages", "<u4"), ("wofs", "<u8"), ("phase", "<u4"),
                        ("reserved", "<u4")])
assert INSTR_DTYPE.itemsize == 64


class MkError(RuntimeError):
    def __init__(self, code, what):
        self.code = code
        super().__init__("%s: %s (%d)" % (what, ERRORS.get(code, "?"), code))


_lib = None


def lib():
    global _lib
    if _lib is None:
        if not os.path.exists(LIB):
            raise ImportError("libmk.so is not built (%s); run __graft_entry__.build()" % LIB)
        L = ctypes.CDLL(LIB)
        P = _vp
        sig = {
            "mk_error_string": (ctypes.c_char_p, [ctypes.c_int]),
            "mk_plan": (ctypes.c_int, [ctypes.POINTER(mk_config), ctypes.POINTER(P)]),
            "mk_plan_info": (ctypes.c_int, [P, ctypes.POINTER(mk_plan_info_t)]),
            "mk_plan_tables": (ctypes.c_int, [P, ctypes.POINTER(P), ctypes.POINTER(ctypes.c_size_t),
                                              ctypes.POINTER(P), ctypes.POINTER(ctypes.c_size_t)]),
            "mk_plan_phases": (ctypes.c_int, [P, ctypes.POINTER(P), ctypes.POINTER(ctypes.c_size_t)]),
            "mk_plan_lists": (ctypes.c_int, [P, ctypes.POINTER(P), ctypes.POINTER(P),
                                             ctypes.POINTER(ctypes.c_size_t)]),
            "mk_load_weights": (ctypes.c_int, [P, ctypes.POINTER(mk_weights), P]),
            "mk_decode_step": (ctypes.c_int, [P, P, P, ctypes.POINTER(mk_kv_cache), P, P]),
            "mk_decode_step_host": (ctypes.c_int, [P, P, P, ctypes.POINTER(mk_kv_cache), P, P]),
            "mk_multikernel_step": (ctypes.c_int, [P, P, P, ctypes.POINTER(mk_kv_cache), P,
                                                   ctypes.c_int, P]),
            "mk_run_phase": (ctypes.c_int, [P, ctypes.c_int, P, P, ctypes.POINTER(mk_kv_cache),
                                            P, P]),
            "mk_status": (ctypes.c_int, [P, P]),
            "mk_read_counters": (ctypes.c_int, [P, P, P, P, P]),
            "mk_read_trace": (ctypes.c_int, [P, P]),
            "mk_debug_buffers": (ctypes.c_int, [P, ctypes.POINTER(mk_debug_buffers_t)]),
            "mk_reset": (ctypes.c_int, [P, P]),
            "mk_destroy": (None, [P]),
        }
        for name, (res, args) in sig.items():
            f = getattr(L, name)
            f.restype = res
            f.argtypes = args
        _lib = L
    return _lib


def _check(code, what):
    if code != MK_OK:
        raise MkError(code, what)


def _ptr(x):
    """Address of a torch tensor, numpy array or int (None -> NULL)."""
    if x is None:
        return None
    if isinstance(x, int):
        return x
    if hasattr(x, "data_ptr"):
        return x.data_ptr()
    if isinstance(x, np.ndarray):
        assert x.flags["C_CONTIGUOUS"]
        return x.ctypes.data
    raise TypeError("cannot take the address of %r" % type(x))


def _stream(s):
    if s is None:
        return None
    if isinstance(s, int):
        return s
    return s.cuda_stream  # torch.cuda.Stream


def mk_error_string(code):
    return lib().mk_error_string(code).decode()


def make_config(model, batch, max_ctx, **kw):
    """mk_config from a model-shape dict (keys as in mk_config) plus options."""
    c = mk_config()
    for k in ("n_layers", "hidden", "n_q_heads", "n_kv_heads", "head_dim", "ffn_dim", "vocab"):
        setattr(c, k, int(model[k]))
    c.rms_eps = float(model["rms_eps"])
    c.rope_theta = float(model["rope_theta"])
    c.tie_embeddings = int(kw.pop("tie_embeddings", model.get("tie_embeddings", 0)))
    c.batch = int(batch)
    c.max_ctx = int(max_ctx)
    for k, v in kw.items():
        setattr(c, k, v)
    return c


def mk_plan(cfg):
    h = _vp()
    _check(lib().mk_plan(ctypes.byref(cfg), ctypes.byref(h)), "mk_plan")
    return h


def mk_plan_info(plan):
    info = mk_plan_info_t()
    _check(lib().mk_plan_info(plan, ctypes.byref(info)), "mk_plan_info")
    return {k: getattr(info, k) for k, _ in mk_plan_info_t._fields_}


def mk_plan_tables(plan):
    """(records as a structured numpy array, raw bytes, per-counter increments)"""
    ip, n, cp, nc = _vp(), ctypes.c_size_t(), _vp(), ctypes.c_size_t()
    _check(lib().mk_plan_tables(plan, ctypes.byref(ip), ctypes.byref(n), ctypes.byref(cp),
                                ctypes.byref(nc)), "mk_plan_tables")
    raw = np.ctypeslib.as_array(ctypes.cast(ip, ctypes.POINTER(ctypes.c_uint8)),
                                shape=(n.value * 64,)).copy()
    inc = np.ctypeslib.as_array(ctypes.cast(cp, ctypes.POINTER(ctypes.c_uint32)),
                                shape=(nc.value,)).copy()
    return raw.view(INSTR_DTYPE), raw, inc


def mk_plan_phases(plan):
    pp, n = _vp(), ctypes.c_size_t()
    _check(lib().mk_plan_phases(plan, ctypes.byref(pp), ctypes.byref(n)), "mk_plan_phases")
    arr = ctypes.cast(pp, ctypes.POINTER(mk_phase))
    return [(arr[i].first, arr[i].count, arr[i].op, arr[i].layer) for i in range(n.value)]


def mk_plan_lists(plan):
    op, ip, n = _vp(), _vp(), ctypes.c_size_t()
    _check(lib().mk_plan_lists(plan, ctypes.byref(op), ctypes.byref(ip), ctypes.byref(n)),
           "mk_plan_lists")
    off = np.ctypeslib.as_array(ctypes.cast(op, ctypes.POINTER(ctypes.c_uint32)),
                                shape=(n.value + 1,)).copy()
    idx = np.ctypeslib.as_array(ctypes.cast(ip, ctypes.POINTER(ctypes.c_uint32)),
                                shape=(int(off[-1]),)).copy()
    return off, idx


def mk_load_weights(plan, w, stream=None):
    """w: dict with embed, final_norm, lm_head (None when tied) and layers[l][name],
    each a torch tensor (any device) or numpy uint16 array of bf16 bits."""
    n = len(w["layers"])
    layers = (mk_layer_weights * n)()
    for l, lw in enumerate(w["layers"]):
        for k in LAYER_FIELDS:
            setattr(layers[l], k, _ptr(lw[k]))
    mw = mk_weights(_ptr(w["embed"]), _ptr(w["final_norm"]), _ptr(w.get("lm_head")), layers)
    _check(lib().mk_load_weights(plan, ctypes.byref(mw), _stream(stream)), "mk_load_weights")


def _kv(kv):
    return mk_kv_cache(_ptr(kv[0]), _ptr(kv[1]))


def mk_decode_step(plan, tokens, positions, kv, logits, stream=None):
    k = _kv(kv)
    _check(lib().mk_decode_step(plan, _ptr(tokens), _ptr(positions), ctypes.byref(k),
                                _ptr(logits), _stream(stream)), "mk_decode_step")


def mk_decode_step_host(plan, tokens, positions, kv, logits, stream=None):
    k = _kv(kv)
    _check(lib().mk_decode_step_host(plan, _ptr(tokens), _ptr(positions), ctypes.byref(k),
                                     _ptr(logits), _stream(stream)), "mk_decode_step_host")


def mk_multikernel_step(plan, tokens, positions, kv, logits, use_graph=False, stream=None):
    k = _kv(kv)
    _check(lib().mk_multikernel_step(plan, _ptr(tokens), _ptr(positions), ctypes.byref(k),
                                     _ptr(logits), int(bool(use_graph)), _stream(stream)),
           "mk_multikernel_step")


def mk_run_phase(plan, phase, tokens, positions, kv, logits, stream=None):
    k = _kv(kv)
    _check(lib().mk_run_phase(plan, int(phase), _ptr(tokens), _ptr(positions), ctypes.byref(k),
                              _ptr(logits), _stream(stream)), "mk_run_phase")


def mk_status(plan, stream=None):
    """Returns the latched device code (0 = ok); does not raise for device errors."""
    return lib().mk_status(plan, _stream(stream))


def mk_read_counters(plan):
    info = mk_plan_info(plan)
    ctr = np.zeros(info["n_counters"], np.uint32)
    exe = np.zeros(info["n_instr"], np.uint32)
    q, e = ctypes.c_uint32(), ctypes.c_uint32()
    _check(lib().mk_read_counters(plan, ctr.ctypes.data, ctypes.addressof(q), exe.ctypes.data,
                                  ctypes.addressof(e)), "mk_read_counters")
    return ctr, q.value, exe, e.value


def mk_read_trace(plan):
    info = mk_plan_info(plan)
    tr = np.zeros((info["n_instr"], 10), np.uint64)
    _check(lib().mk_read_trace(plan, tr.ctypes.data), "mk_read_trace")
    return tr


def mk_debug_buffers(plan):
    b = mk_debug_buffers_t()
    _check(lib().mk_debug_buffers(plan, ctypes.byref(b)), "mk_debug_buffers")
    return {k: getattr(b, k) for k, _ in mk_debug_buffers_t._fields_}


def mk_reset(plan, stream=None):
    _check(lib().mk_reset(plan, _stream(stream)), "mk_reset")


def mk_destroy(plan):
    lib().mk_destroy(plan)


def mk_attention_noalloc(q, k_cache, v_cache, positions, out, batch, n_q_heads, n_kv_heads,
                         head_dim, max_ctx, stream=None):
    """Decode attention for callers that cannot allocate device memory: its
    scratch is the library's fixed static device array (see mk.h)."""
    f = lib().mk_attention_noalloc
    f.restype = ctypes.c_int
    f.argtypes = [_vp] * 5 + [_i32] * 5 + [_vp]
    _check(f(_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(positions), _ptr(out), batch,
             n_q_heads, n_kv_heads, head_dim, max_ctx, _stream(stream)), "mk_attention_noalloc")
