"""CPU oracle -- TEST INFRASTRUCTURE ONLY.

A plain, slow, single-threaded fp64 C restatement of a Llama-style decode step
(oracle.c) and an independent replay of the megakernel's instruction table
(replay.c).  Only tests/, __graft_entry__.smoke() and bench.py's CPU-baseline
leg may import this package.  It never imports the CUDA library and shares no
code with it.

Parity pins: every function is pinned by tests/test_oracle_pins.py,
tests/test_fp8_pins.py and tests/test_replay_pins.py against closed forms,
invariants, brute force and independent library routines.
"""
import ctypes
import os

import numpy as np

from ._build import LIB, build

_lib = None
_D = ctypes.POINTER(ctypes.c_double)
_U16 = ctypes.POINTER(ctypes.c_uint16)


Q8_KINDS = ("wq", "wk", "wv", "wo", "w_gate", "w_up", "w_down")


class _Q8(ctypes.Structure):
    # codes per kind (wq ...), then scales per kind (sq ...), then the LM head
    _fields_ = [(k, ctypes.POINTER(ctypes.c_void_p)) for k in Q8_KINDS] + [
        ("s" + k[1:], ctypes.POINTER(ctypes.c_void_p)) for k in Q8_KINDS] + [
        ("lm", ctypes.c_void_p), ("s_lm", ctypes.c_void_p)]


class _Model(ctypes.Structure):
    _fields_ = [("L", ctypes.c_int), ("H", ctypes.c_int), ("nq", ctypes.c_int),
                ("nkv", ctypes.c_int), ("d", ctypes.c_int), ("F", ctypes.c_int),
                ("V", ctypes.c_int), ("eps", ctypes.c_double), ("theta", ctypes.c_double),
                ("embed", ctypes.c_void_p), ("final_norm", ctypes.c_void_p),
                ("lm_head", ctypes.c_void_p)] + [
        (k, ctypes.POINTER(ctypes.c_void_p)) for k in
        ("attn_norm", "wq", "wk", "wv", "wo", "mlp_norm", "w_gate", "w_up", "w_down")] + [
        ("q8", ctypes.POINTER(_Q8))]


class _Shape(ctypes.Structure):
    _fields_ = [(k, ctypes.c_int) for k in ("L", "H", "nq", "nkv", "d", "F", "V", "B")]


def lib():
    global _lib
    if _lib is None:
        if not os.path.exists(LIB):
            build()
        L = ctypes.CDLL(LIB)
        vp, i, dbl = ctypes.c_void_p, ctypes.c_int, ctypes.c_double
        sig = {
            "or_bf16_to_double": (dbl, [ctypes.c_uint16]),
            "or_bf16_rne": (ctypes.c_uint16, [dbl]),
            "or_rmsnorm": (None, [i, vp, vp, dbl, vp]),
            "or_matvec": (None, [i, i, vp, vp, vp]),
            "or_e4m3_to_double": (dbl, [ctypes.c_uint8]),
            "or_e4m3_rne": (ctypes.c_uint8, [dbl]),
            "or_quantize_rows": (None, [i, i, vp, vp, vp]),
            "or_matvec_q8": (None, [i, i, vp, vp, vp, vp]),
            "or_rope": (None, [i, dbl, dbl, vp]),
            "or_silu": (dbl, [dbl]),
            "or_attention": (None, [i, i, vp, vp, vp, vp]),
            "or_argmax": (i, [i, vp]),
            "or_decode_step": (i, [ctypes.POINTER(_Model), i, i, vp, vp, vp, vp, vp]),
            "or_replay": (i, [vp, i, i, ctypes.POINTER(_Shape), i, vp, vp, vp,
                              ctypes.c_char_p, i]),
            "or_simulate": (i, [vp, i, i, i, i, ctypes.c_uint64, i, vp, vp, vp, i, i,
                                ctypes.c_char_p, i]),
            "or_explore": (ctypes.c_long, [vp, i, i, i, ctypes.c_long, ctypes.c_char_p, i]),
            "or_redeal": (i, [vp, i, ctypes.POINTER(_Shape), i, vp, vp, i, vp, ctypes.c_char_p,
                              i]),
        }
        for name, (res, args) in sig.items():
            f = getattr(L, name)
            f.restype = res
            f.argtypes = args
        _lib = L
    return _lib


def _f64(a):
    return np.ascontiguousarray(a, dtype=np.float64)


def _u16(a):
    return np.ascontiguousarray(a, dtype=np.uint16)


def bf16_to_double(h):
    return float(lib().or_bf16_to_double(int(h)))


def bf16_rne(v):
    return int(lib().or_bf16_rne(float(v)))


def rmsnorm(x, g, eps):
    x, g = _f64(x), _u16(g)
    y = np.empty_like(x)
    lib().or_rmsnorm(x.size, x.ctypes.data, g.ctypes.data, eps, y.ctypes.data)
    return y


def matvec(W, x):
    W, x = _u16(W), _f64(x)
    M, K = W.shape
    y = np.empty(M)
    lib().or_matvec(M, K, W.ctypes.data, x.ctypes.data, y.ctypes.data)
    return y


def e4m3_to_double(c):
    return float(lib().or_e4m3_to_double(int(c)))


def e4m3_rne(v):
    return int(lib().or_e4m3_rne(float(v)))


def quantize_rows(W):
    """FP8 form of a bf16 matrix [M][K]: (E4M3 codes uint8 [M][K], float32
    row scales [M])."""
    W = _u16(W)
    M, K = W.shape
    Q = np.empty((M, K), np.uint8)
    s = np.empty(M, np.float32)
    lib().or_quantize_rows(M, K, W.ctypes.data, Q.ctypes.data, s.ctypes.data)
    return Q, s


def matvec_q8(Q, s, x):
    Q, s, x = np.ascontiguousarray(Q, np.uint8), np.ascontiguousarray(s, np.float32), _f64(x)
    M, K = Q.shape
    y = np.empty(M)
    lib().or_matvec_q8(M, K, Q.ctypes.data, s.ctypes.data, x.ctypes.data, y.ctypes.data)
    return y


def rope(z, pos, theta):
    z = _f64(z).copy()
    lib().or_rope(z.size, float(pos), float(theta), z.ctypes.data)
    return z


def silu(z):
    return float(lib().or_silu(float(z)))


def attention(q, K, V):
    q, K, V = _f64(q), _u16(K), _u16(V)
    n, d = K.shape
    o = np.empty(d)
    lib().or_attention(d, n, q.ctypes.data, K.ctypes.data, V.ctypes.data, o.ctypes.data)
    return o


def argmax(v):
    v = _f64(v)
    return int(lib().or_argmax(v.size, v.ctypes.data))


class Model:
    """Holds a model's bf16 weights (numpy uint16, PyTorch layout) and its own
    KV cache, and runs oracle decode steps on them."""

    def __init__(self, cfg, weights, batch, max_ctx, kcache, vcache, fp8=False):
        """fp8: every projection and the LM head in their FP8 form
        (quantize_rows); the token lookup and the norms stay bf16."""
        self.cfg, self.w, self.B, self.max_ctx = cfg, weights, batch, max_ctx
        self.k = np.array(kcache, dtype=np.uint16, copy=True, order="C")
        self.v = np.array(vcache, dtype=np.uint16, copy=True, order="C")
        L = cfg["n_layers"]
        self._keep = []

        def arr(kind):
            ptrs = (ctypes.c_void_p * L)(*[weights["layers"][l][kind].ctypes.data
                                           for l in range(L)])
            self._keep.append(ptrs)
            return ctypes.cast(ptrs, ctypes.POINTER(ctypes.c_void_p))

        m = _Model()
        m.L, m.H, m.nq, m.nkv = L, cfg["hidden"], cfg["n_q_heads"], cfg["n_kv_heads"]
        m.d, m.F, m.V = cfg["head_dim"], cfg["ffn_dim"], cfg["vocab"]
        m.eps, m.theta = cfg["rms_eps"], cfg["rope_theta"]
        m.embed = weights["embed"].ctypes.data
        m.final_norm = weights["final_norm"].ctypes.data
        m.lm_head = weights["lm_head"].ctypes.data if weights["lm_head"] is not None else None
        for kind in ("attn_norm", "wq", "wk", "wv", "wo", "mlp_norm", "w_gate", "w_up",
                     "w_down"):
            setattr(m, kind, arr(kind))
        if fp8:
            q8 = _Q8()
            for kind in Q8_KINDS:
                sk = "s" + kind[1:]
                qs = [quantize_rows(weights["layers"][l][kind]) for l in range(L)]
                self._keep.append(qs)
                for field, j in ((kind, 0), (sk, 1)):
                    ptrs = (ctypes.c_void_p * L)(*[qs[l][j].ctypes.data for l in range(L)])
                    self._keep.append(ptrs)
                    setattr(q8, field, ctypes.cast(ptrs, ctypes.POINTER(ctypes.c_void_p)))
            lm = weights["lm_head"] if weights["lm_head"] is not None else weights["embed"]
            self.q8_lm = quantize_rows(lm)
            q8.lm, q8.s_lm = self.q8_lm[0].ctypes.data, self.q8_lm[1].ctypes.data
            self._q8 = q8
            m.q8 = ctypes.pointer(q8)
        self._m = m

    def step(self, tokens, positions):
        tokens = np.ascontiguousarray(tokens, dtype=np.int32)
        positions = np.ascontiguousarray(positions, dtype=np.int32)
        assert tokens.shape == (self.B,) and positions.shape == (self.B,)
        logits = np.empty((self.B, self.cfg["vocab"]))
        rc = lib().or_decode_step(ctypes.byref(self._m), self.B, self.max_ctx,
                                  self.k.ctypes.data, self.v.ctypes.data, tokens.ctypes.data,
                                  positions.ctypes.data, logits.ctypes.data)
        if rc != 0:
            raise ValueError("oracle step rejected its arguments")
        return logits


def replay(table, n_instr, n_counters, cfg, batch, n_sms, list_off=None, list_idx=None):
    """Check an instruction table; returns the per-step signal count of every
    counter (uint32 array).  Raises AssertionError with the reason on failure."""
    table = np.ascontiguousarray(table, dtype=np.uint8)
    assert table.size == 64 * n_instr
    s = _Shape(cfg["n_layers"], cfg["hidden"], cfg["n_q_heads"], cfg["n_kv_heads"],
               cfg["head_dim"], cfg["ffn_dim"], cfg["vocab"], batch)
    inc = np.zeros(n_counters, dtype=np.uint32)
    msg = ctypes.create_string_buffer(512)
    lo = None if list_off is None else np.ascontiguousarray(list_off, dtype=np.uint32)
    li = None if list_idx is None else np.ascontiguousarray(list_idx, dtype=np.uint32)
    rc = lib().or_replay(table.ctypes.data, n_instr, n_counters, ctypes.byref(s), n_sms,
                         None if lo is None else lo.ctypes.data,
                         None if li is None else li.ctypes.data, inc.ctypes.data, msg, 512)
    if rc != 0:
        raise AssertionError("replay: " + msg.value.decode())
    return inc


def simulate(table, n_instr, n_counters, n_sms, fifo_depth, seed=0, trials=4, list_off=None,
             list_idx=None, att_first=None, att_count=0):
    """Seeded random interleavings of n_sms virtual SMs (dynamic queue, static
    lists, or hybrid lists whose marker entries claim from per-layer attention
    queues: att_first[l] + 0 .. att_count - 1).  Raises on a deadlock."""
    table = np.ascontiguousarray(table, dtype=np.uint8)
    msg = ctypes.create_string_buffer(512)
    lo = None if list_off is None else np.ascontiguousarray(list_off, dtype=np.uint32)
    li = None if list_idx is None else np.ascontiguousarray(list_idx, dtype=np.uint32)
    af = None if att_first is None else np.ascontiguousarray(att_first, dtype=np.uint32)
    rc = lib().or_simulate(table.ctypes.data, n_instr, n_counters, n_sms, fifo_depth, seed,
                           trials, None if lo is None else lo.ctypes.data,
                           None if li is None else li.ctypes.data,
                           None if af is None else af.ctypes.data,
                           0 if af is None else af.size, int(att_count), msg, 512)
    if rc != 0:
        raise AssertionError("simulate: " + msg.value.decode())


def explore(table, n_instr, n_counters, fifo_depth, max_states=2_000_000):
    table = np.ascontiguousarray(table, dtype=np.uint8)
    msg = ctypes.create_string_buffer(512)
    n = lib().or_explore(table.ctypes.data, n_instr, n_counters, fifo_depth, max_states, msg, 512)
    if n < 0:
        raise AssertionError("explore: " + msg.value.decode())
    return n


def redeal(table, n_instr, cfg, batch, attn_chunk, positions, list_idx=None):
    """Executed instruction of every list slot (uint32 array, the order of
    list_idx, or of the queue when list_idx is None) once each batched
    attention phase is re-dealt for `positions`: chunks with work first.
    Raises AssertionError when the table does not allow the re-deal."""
    table = np.ascontiguousarray(table, dtype=np.uint8)
    assert table.size == 64 * n_instr
    s = _Shape(cfg["n_layers"], cfg["hidden"], cfg["n_q_heads"], cfg["n_kv_heads"],
               cfg["head_dim"], cfg["ffn_dim"], cfg["vocab"], batch)
    pos = np.ascontiguousarray(positions, dtype=np.int32)
    assert pos.size == batch
    li = None if list_idx is None else np.ascontiguousarray(list_idx, dtype=np.uint32)
    out = np.zeros(n_instr, dtype=np.uint32)
    msg = ctypes.create_string_buffer(512)
    rc = lib().or_redeal(table.ctypes.data, n_instr, ctypes.byref(s), int(attn_chunk),
                         pos.ctypes.data, None if li is None else li.ctypes.data, n_instr,
                         out.ctypes.data, msg, 512)
    if rc != 0:
        raise AssertionError("redeal: " + msg.value.decode())
    return out
