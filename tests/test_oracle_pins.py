"""Pins of the CPU oracle against things other than itself: closed forms,
invariants, exact rational arithmetic, brute force and independent library
routines (torch CPU in float64).  A dropped term, a wrong sign or index or a
transposed operand in oracle.c fails at least one of these."""
import math
import os
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle
import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
rng = np.random.default_rng(1234)


def rand_bf16(shape, std=1.0):
    return synth.f32_to_bf16(rng.normal(0, std, size=shape).astype(np.float32))


def bf(a):
    return synth.bf16_to_f32(a).astype(np.float64)


# ---------------------------------------------------------------- bf16 ----
def test_bf16_patterns_golden():
    for line in open(os.path.join(GOLDEN, "bf16_patterns.txt")):
        if line.startswith("#") or not line.strip():
            continue
        val, bits = line.split()
        assert oracle.bf16_rne(float(val)) == int(bits, 16), line
        if float(val) == oracle.bf16_to_double(int(bits, 16)):
            assert oracle.bf16_to_double(int(bits, 16)) == float(val)


def test_bf16_rne_matches_torch_on_float32_values():
    x = rng.normal(0, 3, size=20000).astype(np.float32)
    x[:50] = np.float32(1.0) + np.arange(50, dtype=np.float32) * np.float32(2.0 ** -9)
    want = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    got = np.array([oracle.bf16_rne(float(v)) for v in x], dtype=np.uint16)
    assert np.array_equal(got, want)


def test_bf16_rne_is_nearest_for_doubles():
    # the oracle rounds doubles directly; no neighbouring pattern is closer
    for v in rng.normal(0, 1, size=3000):
        h = oracle.bf16_rne(v)
        r = oracle.bf16_to_double(h)
        for nb in (h - 1, h + 1):
            if 0 < (nb & 0x7FFF) < 0x7F80:
                assert abs(oracle.bf16_to_double(nb) - v) >= abs(r - v)


# ------------------------------------------------------------- RMSNorm ----
def test_rmsnorm_constant_vector_closed_form():
    n, c, eps = 64, 0.75, 1e-5
    g = rand_bf16(n)
    y = oracle.rmsnorm(np.full(n, c), g, eps)
    want = bf(g) * c / math.sqrt(c * c + eps)
    assert np.allclose(y, want, rtol=1e-14, atol=0)


def test_rmsnorm_unit_gain_gives_unit_rms():
    x = rng.normal(0, 5, size=513)
    ones = np.full(513, 0x3F80, dtype=np.uint16)
    y = oracle.rmsnorm(x, ones, 0.0)
    assert abs(math.sqrt(np.mean(y * y)) - 1.0) < 1e-14


def test_rmsnorm_scale_invariance_and_eps_placement():
    x = rng.normal(0, 1, size=256)
    g = rand_bf16(256)
    a = oracle.rmsnorm(x, g, 0.0)
    b = oracle.rmsnorm(37.5 * x, g, 0.0)
    assert np.allclose(a, b, rtol=1e-13)
    # eps goes inside the square root: for x = 0 except one entry
    x = np.zeros(4)
    x[1] = 2.0
    y = oracle.rmsnorm(x, np.full(4, 0x3F80, dtype=np.uint16), 0.5)
    assert y[1] == pytest.approx(2.0 / math.sqrt(4.0 / 4 + 0.5), rel=1e-15)


def test_rmsnorm_matches_torch():
    x = rng.normal(0, 2, size=2048)
    g = rand_bf16(2048, 0.5)
    y = oracle.rmsnorm(x, g, 1e-5)
    want = torch.nn.functional.rms_norm(torch.from_numpy(x), (2048,),
                                        torch.from_numpy(bf(g)), eps=1e-5).numpy()
    assert np.allclose(y, want, rtol=1e-12, atol=1e-14)


# -------------------------------------------------------------- matvec ----
def test_matvec_exact_rational_bound():
    M, K = 7, 300
    W = rand_bf16((M, K))
    x = rng.normal(0, 1, size=K)
    y = oracle.matvec(W, x)
    wf = bf(W)
    for r in range(M):
        exact = sum(Fraction(float(wf[r, k])) * Fraction(float(x[k])) for k in range(K))
        bound = K * 2.0 ** -53 * float(np.sum(np.abs(wf[r]) * np.abs(x))) * 1.01
        assert abs(Fraction(float(y[r])) - exact) <= Fraction(bound)


def test_matvec_orientation_and_rows():
    # W [out, in]: a single 1 at (r, k) selects x[k] into y[r]
    W = np.zeros((5, 9), dtype=np.uint16)
    W[3, 7] = 0x3F80
    W[0, 2] = 0xC000  # -2
    x = np.arange(9, dtype=np.float64) + 1
    y = oracle.matvec(W, x)
    assert list(y) == [-6.0, 0.0, 0.0, 8.0, 0.0]


def test_matvec_matches_torch():
    W = rand_bf16((64, 1024), 0.02)
    x = rng.normal(0, 1, size=1024)
    want = torch.nn.functional.linear(torch.from_numpy(x), torch.from_numpy(bf(W))).numpy()
    assert np.allclose(oracle.matvec(W, x), want, rtol=1e-12, atol=1e-14)


# ---------------------------------------------------------------- RoPE ----
@pytest.mark.parametrize("d", [2, 64, 128])
def test_rope_preserves_pair_norms_and_identity_at_zero(d):
    z = rng.normal(0, 1, size=d)
    assert np.array_equal(oracle.rope(z, 0, 10000.0), z)
    r = oracle.rope(z, 777, 500000.0)
    h = d // 2
    assert np.allclose(r[:h] ** 2 + r[h:] ** 2, z[:h] ** 2 + z[h:] ** 2, rtol=1e-12)


def test_rope_relative_position_property():
    d, theta = 64, 10000.0
    q, k = rng.normal(size=d), rng.normal(size=d)
    base = np.dot(oracle.rope(q, 10, theta), oracle.rope(k, 3, theta))
    for p, pk in [(17, 10), (1007, 1000), (7, 0)]:
        assert np.dot(oracle.rope(q, p, theta), oracle.rope(k, pk, theta)) == pytest.approx(base, rel=1e-9)


def test_rope_rotate_half_pairing_and_direction():
    # d = 2: one pair (z0, z1) rotated by pos radians counter-clockwise
    r = oracle.rope(np.array([1.0, 0.0]), math.pi / 2, 10000.0)
    assert np.allclose(r, [0.0, 1.0], atol=1e-15)
    # d = 4, theta = 16: pairs (0,2) by pos, (1,3) by pos/4
    r = oracle.rope(np.array([1.0, 1.0, 0.0, 0.0]), math.pi, 16.0)
    assert np.allclose(r, [-1.0, math.cos(math.pi / 4), 0.0, math.sin(math.pi / 4)], atol=1e-15)


def test_rope_matches_complex_formulation():
    d, theta, pos = 128, 500000.0, 8191
    z = rng.normal(size=d)
    h = d // 2
    c = (z[:h] + 1j * z[h:]) * np.exp(1j * pos * theta ** (-2.0 * np.arange(h) / d))
    want = np.concatenate([c.real, c.imag])
    assert np.allclose(oracle.rope(z, pos, theta), want, rtol=1e-10, atol=1e-12)


# ---------------------------------------------------------------- SiLU ----
def test_silu_closed_forms():
    assert oracle.silu(0.0) == 0.0
    assert oracle.silu(40.0) == pytest.approx(40.0, rel=1e-15)
    assert abs(oracle.silu(-40.0)) < 1e-15
    for z in rng.normal(0, 4, size=50):
        assert oracle.silu(z) - oracle.silu(-z) == pytest.approx(z, rel=1e-12, abs=1e-15)
    z = torch.linspace(-9, 9, 101, dtype=torch.float64)
    want = torch.nn.functional.silu(z).numpy()
    got = np.array([oracle.silu(float(v)) for v in z])
    assert np.allclose(got, want, rtol=1e-14, atol=1e-16)


# ----------------------------------------------------------- attention ----
def test_attention_single_key_returns_its_value():
    d = 64
    K, V = rand_bf16((1, d)), rand_bf16((1, d))
    o = oracle.attention(rng.normal(size=d), K, V)
    assert np.allclose(o, bf(V[0]), rtol=1e-15)


def test_attention_equal_scores_average_values():
    d, n = 64, 37
    K, V = rand_bf16((n, d)), rand_bf16((n, d))
    o = oracle.attention(np.zeros(d), K, V)
    assert np.allclose(o, bf(V).mean(axis=0), rtol=1e-12)


def test_attention_weights_sum_to_one():
    d, n = 128, 300
    K = rand_bf16((n, d))
    ones = np.full((n, d), 0x3F80, dtype=np.uint16)
    o = oracle.attention(rng.normal(0, 3, size=d), K, ones)
    assert np.allclose(o, 1.0, rtol=1e-13)


def test_attention_one_hot_selection_by_scale():
    # a huge score on key 5 selects its value; the 1/sqrt(d) scale is applied
    d, n = 64, 9
    K = np.zeros((n, d), dtype=np.uint16)
    K[5, 0] = synth.f32_to_bf16(np.array([8.0], dtype=np.float32))[0]
    V = rand_bf16((n, d))
    q = np.zeros(d)
    q[0] = 100.0
    o = oracle.attention(q, K, V)
    assert np.allclose(o, bf(V[5]), rtol=1e-12)
    # moderate scores: weights are exp(s_j) / sum with s_j = q.k_j / 8
    q[0] = 2.0
    s = np.zeros(n)
    s[5] = 2.0 * 8.0 / 8.0
    p = np.exp(s) / np.exp(s).sum()
    assert np.allclose(oracle.attention(q, K, V), p @ bf(V), rtol=1e-13)


def test_attention_matches_torch_sdpa():
    for d, n in [(64, 1), (64, 65), (128, 200)]:
        q = rng.normal(size=d)
        K, V = rand_bf16((n, d)), rand_bf16((n, d))
        want = torch.nn.functional.scaled_dot_product_attention(
            torch.from_numpy(q)[None, None, None], torch.from_numpy(bf(K))[None, None],
            torch.from_numpy(bf(V))[None, None])[0, 0, 0].numpy()
        assert np.allclose(oracle.attention(q, K, V), want, rtol=1e-12, atol=1e-14)


def test_argmax_ties_lowest_index():
    assert oracle.argmax([1.0, 3.0, 3.0, 2.0]) == 1
    assert oracle.argmax([5.0]) == 0
    assert oracle.argmax([-1.0, -1.0]) == 0


# ---------------------------------------------------- whole decode step ----
def tiny_cfg(**kw):
    c = dict(n_layers=2, hidden=64, n_q_heads=4, n_kv_heads=2, head_dim=16, ffn_dim=96,
             vocab=50, rms_eps=1e-5, rope_theta=10000.0, tie_embeddings=0)
    c.update(kw)
    return c


def rand_model(c, std=0.2, tie=False):
    from synth.workloads import shapes
    w = {"embed": rand_bf16((c["vocab"], c["hidden"]), std),
         "final_norm": synth.f32_to_bf16((1 + rng.normal(0, 0.1, c["hidden"])).astype(np.float32)),
         "lm_head": None if tie else rand_bf16((c["vocab"], c["hidden"]), std),
         "layers": []}
    for _ in range(c["n_layers"]):
        layer = {}
        for k, s in shapes(c).items():
            if k.endswith("norm"):
                layer[k] = synth.f32_to_bf16((1 + rng.normal(0, 0.1, s)).astype(np.float32))
            else:
                layer[k] = rand_bf16(s, std)
        w["layers"].append(layer)
    return w


def torch_reference_step(c, w, kc, vc, tokens, positions):
    """Independent float64 restatement with torch library routines (F.rms_norm,
    F.linear, scaled_dot_product_attention with repeat_interleave for GQA,
    F.silu) and complex-number RoPE; updates kc/vc (torch uint16 views)."""
    F_ = torch.nn.functional
    t = lambda a: torch.from_numpy(bf(a))
    H, nq, nkv, d = c["hidden"], c["n_q_heads"], c["n_kv_heads"], c["head_dim"]
    out = []
    for b, (tok, p) in enumerate(zip(tokens, positions)):
        x = t(w["embed"])[tok]
        for l, lw in enumerate(w["layers"]):
            y = F_.rms_norm(x, (H,), t(lw["attn_norm"]), eps=c["rms_eps"])
            q = F_.linear(y, t(lw["wq"])).view(nq, d)
            k = F_.linear(y, t(lw["wk"])).view(nkv, d)
            v = F_.linear(y, t(lw["wv"])).view(nkv, d)
            h = d // 2
            rot = torch.exp(1j * p * torch.tensor(c["rope_theta"], dtype=torch.float64) **
                            (-2.0 * torch.arange(h, dtype=torch.float64) / d))

            def rope(z):
                zc = torch.complex(z[..., :h], z[..., h:]) * rot
                return torch.cat([zc.real, zc.imag], dim=-1)
            q, k = rope(q), rope(k)
            kc[l, b, :, p] = [[oracle.bf16_rne(float(e)) for e in row] for row in k.numpy()]
            vc[l, b, :, p] = [[oracle.bf16_rne(float(e)) for e in row] for row in v.numpy()]
            Kt = torch.from_numpy(bf(kc[l, b, :, :p + 1]))  # [nkv, p+1, d]
            Vt = torch.from_numpy(bf(vc[l, b, :, :p + 1]))
            Kt = Kt.repeat_interleave(nq // nkv, dim=0)
            Vt = Vt.repeat_interleave(nq // nkv, dim=0)
            o = F_.scaled_dot_product_attention(q[:, None, :], Kt, Vt)[:, 0, :].reshape(-1)
            x = x + F_.linear(o, t(lw["wo"]))
            y = F_.rms_norm(x, (H,), t(lw["mlp_norm"]), eps=c["rms_eps"])
            x = x + F_.linear(F_.silu(F_.linear(y, t(lw["w_gate"]))) * F_.linear(y, t(lw["w_up"])),
                              t(lw["w_down"]))
        y = F_.rms_norm(x, (H,), t(w["final_norm"]), eps=c["rms_eps"])
        lm = w["lm_head"] if w["lm_head"] is not None else w["embed"]
        out.append(F_.linear(y, t(lm)).numpy())
    return np.stack(out)


@pytest.mark.parametrize("tie", [False, True])
def test_decode_step_matches_torch_restatement(tie):
    c = tiny_cfg()
    w = rand_model(c, tie=tie)
    B, mctx = 2, 32
    ctx = [5, 11]
    kc = np.zeros((c["n_layers"], B, c["n_kv_heads"], mctx, c["head_dim"]), dtype=np.uint16)
    vc = np.zeros_like(kc)
    for b in range(B):
        kc[:, b, :, :ctx[b]] = rand_bf16(kc[:, b, :, :ctx[b]].shape)
        vc[:, b, :, :ctx[b]] = rand_bf16(vc[:, b, :, :ctx[b]].shape)
    m = oracle.Model(c, w, B, mctx, kc, vc)
    kr, vr = kc.copy(), vc.copy()
    for step in range(3):
        toks = np.array([7 + step, 31 - step], dtype=np.int32)
        pos = np.array(ctx, dtype=np.int32) + step
        got = m.step(toks, pos)
        want = torch_reference_step(c, w, kr, vr, toks, pos)
        assert np.allclose(got, want, rtol=1e-10, atol=1e-11)
        # the oracle's cache holds bf16 of its own k/v; the restatement rounds
        # its own values; they may differ by a rounding-boundary ulp at most
        diff = np.abs(synth.bf16_to_f32(m.k).astype(np.float64) - synth.bf16_to_f32(kr))
        assert diff.max() <= 2 ** -6 * max(1.0, np.abs(synth.bf16_to_f32(kr)).max())


def test_zero_layer_model_closed_form():
    c = tiny_cfg(n_layers=0)
    w = rand_model(c)
    m = oracle.Model(c, w, 1, 8, np.zeros((0, 1, 2, 8, 16), np.uint16),
                     np.zeros((0, 1, 2, 8, 16), np.uint16))
    got = m.step([13], [0])[0]
    x = bf(w["embed"][13])
    y = x / math.sqrt(np.mean(x * x) + c["rms_eps"]) * bf(w["final_norm"])
    assert np.allclose(got, bf(w["lm_head"]) @ y, rtol=1e-12, atol=1e-14)


def test_pass_through_layers_keep_the_residual_and_append_kv():
    # Wo = Wd = 0: every layer leaves x unchanged but still writes K/V at p
    c = tiny_cfg()
    w = rand_model(c)
    for lw in w["layers"]:
        lw["wo"][:] = 0
        lw["w_down"][:] = 0
    kc = np.zeros((2, 1, 2, 16, 16), np.uint16)
    m = oracle.Model(c, w, 1, 16, kc, kc)
    got = m.step([3], [9])[0]
    x = bf(w["embed"][3])
    y = x / math.sqrt(np.mean(x * x) + c["rms_eps"]) * bf(w["final_norm"])
    assert np.allclose(got, bf(w["lm_head"]) @ y, rtol=1e-12, atol=1e-14)
    for l in range(2):
        yl = x / math.sqrt(np.mean(x * x) + c["rms_eps"]) * bf(w["layers"][l]["attn_norm"])
        v = bf(w["layers"][l]["wv"]) @ yl
        for g in range(2):
            want = [oracle.bf16_rne(e) for e in v[16 * g:16 * (g + 1)]]
            assert list(m.v[l, 0, g, 9]) == want
        assert not m.k[l, 0, :, 10:].any() and not m.k[l, 0, :, :9].any()


def test_uniform_attention_hand_case():
    # Wq = 0 makes every score equal: attention is the mean of V[0..p]
    # (including the value written at p); Wv = Wo = identity and a zero MLP
    # give x' = x + mean(V), checkable by hand.
    c = tiny_cfg(n_layers=1, hidden=16, n_q_heads=1, n_kv_heads=1, head_dim=16, ffn_dim=8,
                 vocab=6)
    w = rand_model(c)
    lw = w["layers"][0]
    lw["wq"][:] = 0
    eye = np.zeros((16, 16), np.uint16)
    eye[np.arange(16), np.arange(16)] = 0x3F80
    lw["wv"][:] = eye
    lw["wo"][:] = eye
    lw["w_down"][:] = 0
    p = 3
    kc = np.zeros((1, 1, 1, 8, 16), np.uint16)
    vc = np.zeros_like(kc)
    vc[0, 0, 0, :p] = rand_bf16((p, 16))
    m = oracle.Model(c, w, 1, 8, kc, vc)
    got = m.step([2], [p])[0]
    x = bf(w["embed"][2])
    y1 = x / math.sqrt(np.mean(x * x) + c["rms_eps"]) * bf(lw["attn_norm"])
    vnew = bf(np.array([oracle.bf16_rne(e) for e in y1], np.uint16))
    mean_v = (bf(vc[0, 0, 0, :p]).sum(axis=0) + vnew) / (p + 1)
    x2 = x + mean_v
    yf = x2 / math.sqrt(np.mean(x2 * x2) + c["rms_eps"]) * bf(w["final_norm"])
    assert np.allclose(got, bf(w["lm_head"]) @ yf, rtol=1e-12, atol=1e-14)


def test_gqa_grouping_is_contiguous():
    # q heads 0,1 use kv group 0 and heads 2,3 use group 1 (HF repeat_kv)
    c = tiny_cfg(n_layers=1)
    w = rand_model(c)
    lw = w["layers"][0]
    for k in ("w_gate", "w_up", "w_down"):
        lw[k][:] = 0
    kc = np.zeros((1, 1, 2, 8, 16), np.uint16)
    vc = np.zeros_like(kc)
    vc[0, 0, 1, :4] = rand_bf16((4, 16))  # only group 1 has values
    lw["wv"][:] = 0                        # and the new value is zero
    m = oracle.Model(c, w, 1, 8, kc, vc)
    # with only Wo columns of heads 0,1 non-zero, group 1 must not leak in
    wo = lw["wo"].copy()
    lw["wo"][:, 32:] = 0
    a = oracle.Model(c, w, 1, 8, kc, vc).step([1], [4])[0]
    lw["wo"][:] = 0
    b = oracle.Model(c, w, 1, 8, kc, vc).step([1], [4])[0]
    assert np.allclose(a, b, rtol=1e-13)
    lw["wo"][:] = wo
    lw["wo"][:, :32] = 0
    c2 = oracle.Model(c, w, 1, 8, kc, vc).step([1], [4])[0]
    assert not np.allclose(c2, b)
    del m


def test_out_of_range_arguments_are_rejected():
    c = tiny_cfg(n_layers=1)
    w = rand_model(c)
    kc = np.zeros((1, 1, 2, 8, 16), np.uint16)
    m = oracle.Model(c, w, 1, 8, kc, kc)
    with pytest.raises(ValueError):
        m.step([c["vocab"]], [0])
    with pytest.raises(ValueError):
        m.step([0], [8])
