"""Pins of the oracle's FP8 weight form (E4M3 codes with one scale per output
row) against things other than itself: the format's defining values, brute
force over all 256 codes, torch's float8_e4m3fn conversion (a library
routine) on in-range values, and an exactness identity for the whole decode
step.  A wrong exponent bias, mantissa width, rounding direction, saturation
or scale placement fails at least one of these."""
import math

import numpy as np
import pytest
import torch

import oracle
import synth

rng = np.random.default_rng(4321)
FINITE = [c for c in range(256) if c & 0x7F != 0x7F]  # every code but the two NaNs


def test_e4m3_defining_values():
    # sign, 4 exponent bits (bias 7), 3 mantissa bits; field 0 subnormal
    want = {0x00: 0.0, 0x01: 2.0 ** -9, 0x07: 7 * 2.0 ** -9, 0x08: 2.0 ** -6,
            0x38: 1.0, 0x39: 1.125, 0x3F: 1.875, 0x40: 2.0, 0x77: 240.0, 0x78: 256.0,
            0x7E: 448.0, 0x81: -(2.0 ** -9), 0xB8: -1.0, 0xFE: -448.0}
    for c, v in want.items():
        assert oracle.e4m3_to_double(c) == v, hex(c)
    assert math.copysign(1.0, oracle.e4m3_to_double(0x80)) == -1.0
    assert math.isnan(oracle.e4m3_to_double(0x7F)) and math.isnan(oracle.e4m3_to_double(0xFF))


def test_e4m3_round_trip_of_every_finite_code():
    for c in FINITE:
        assert oracle.e4m3_rne(oracle.e4m3_to_double(c)) == c, hex(c)


def test_e4m3_rounding_ties_and_saturation():
    assert oracle.e4m3_rne(1.0625) == 0x38        # halfway 1 / 1.125 -> even (1)
    assert oracle.e4m3_rne(1.1875) == 0x3A        # halfway 1.125 / 1.25 -> even (1.25)
    assert oracle.e4m3_rne(2.0 ** -10) == 0x00    # half the smallest subnormal -> 0
    assert oracle.e4m3_rne(3 * 2.0 ** -10) == 0x02  # halfway codes 1 / 2 -> even
    assert oracle.e4m3_rne(15.5 * 2.0 ** -10) == 0x08  # rounds up out of the subnormals
    assert oracle.e4m3_rne(1.96875) == 0x40       # 1.9375 halfway to 2 rounds up a binade
    assert oracle.e4m3_rne(440.0) == 0x7E         # nearer 448 than 416
    assert oracle.e4m3_rne(1e6) == 0x7E and oracle.e4m3_rne(-1e6) == 0xFE  # saturate
    assert oracle.e4m3_rne(-0.0) == 0x80


def test_e4m3_is_the_nearest_code_by_brute_force():
    vals = np.array([oracle.e4m3_to_double(c) for c in FINITE])
    xs = np.concatenate([rng.uniform(-448, 448, 400),
                         np.exp2(rng.uniform(-12, 8.8, 400)) * rng.choice([-1, 1], 400)])
    for x in xs:
        got = oracle.e4m3_to_double(oracle.e4m3_rne(x))
        assert abs(got - x) <= np.min(np.abs(vals - x)) + 0.0, x


def test_e4m3_matches_torch_float8_on_in_range_values():
    xs = np.concatenate([rng.uniform(-447, 447, 2000),
                         np.exp2(rng.uniform(-12, 8.7, 2000)) * rng.choice([-1, 1], 2000)])
    xs = xs.astype(np.float32)
    want = torch.from_numpy(xs).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = np.array([oracle.e4m3_rne(float(x)) for x in xs], np.uint8)
    assert np.array_equal(got, want)


def test_quantize_rows_scale_and_extremes():
    W = synth.f32_to_bf16(rng.normal(0, 0.02, (6, 96)).astype(np.float32))
    W[3] = 0                                    # a zero row: scale 1, all codes 0
    Q, s = oracle.quantize_rows(W)
    Wf = synth.bf16_to_f32(W)
    for r in range(6):
        amax = np.float32(np.abs(Wf[r]).max())
        if r == 3:
            assert s[r] == 1.0 and not Q[r].any()
            continue
        assert s[r] == np.float32(amax / np.float32(448.0))
        k = int(np.argmax(np.abs(Wf[r])))
        assert Q[r, k] in (0x7E, 0xFE)          # the row's largest magnitude -> +-448
        deq = np.array([oracle.e4m3_to_double(c) for c in Q[r]]) * float(s[r])
        normal = np.abs(Wf[r]) >= 2.0 ** -6 * s[r]
        rel = np.abs(deq - Wf[r])[normal] / np.abs(Wf[r])[normal]
        assert rel.max() <= 2.0 ** -4            # 3 mantissa bits: half an ulp
        assert np.array_equal(np.sign(deq[normal]), np.sign(Wf[r][normal]))


def test_matvec_q8_brute_force():
    Q = rng.integers(0, 256, (5, 40)).astype(np.uint8)
    Q[(Q & 0x7F) == 0x7F] = 0x38                 # no NaN codes
    s = rng.uniform(0.01, 2.0, 5).astype(np.float32)
    x = rng.normal(size=40)
    want = np.array([sum(oracle.e4m3_to_double(Q[r, k]) * float(s[r]) * x[k] for k in range(40))
                     for r in range(5)])
    assert np.allclose(oracle.matvec_q8(Q, s, x), want, rtol=1e-13, atol=1e-13)


def exact_fp8_model(c, tie):
    """bf16 weights whose FP8 form is exact: every row holds E4M3 values times
    a power of two, its largest magnitude exactly 448 times that power, so
    scale = a power of two and code * scale = the bf16 weight."""
    from synth.workloads import shapes

    def mat(shape):
        M, K = shape
        codes = rng.choice(FINITE, size=(M, K))
        v = np.array([[oracle.e4m3_to_double(q) for q in row] for row in codes])
        v[:, 0] = 448.0 * rng.choice([-1, 1], M)
        v *= np.exp2(rng.integers(-12, -6, (M, 1)))
        return synth.f32_to_bf16(v.astype(np.float32))
    w = {"embed": mat((c["vocab"], c["hidden"])),
         "final_norm": synth.f32_to_bf16((1 + rng.normal(0, 0.1, c["hidden"])).astype(np.float32)),
         "lm_head": None if tie else mat((c["vocab"], c["hidden"])), "layers": []}
    for _ in range(c["n_layers"]):
        layer = {}
        for k, s in shapes(c).items():
            layer[k] = (synth.f32_to_bf16((1 + rng.normal(0, 0.1, s)).astype(np.float32))
                        if k.endswith("norm") else mat(s))
        w["layers"].append(layer)
    return w


@pytest.mark.parametrize("tie", [False, True])
def test_fp8_decode_step_equals_bf16_step_when_the_fp8_form_is_exact(tie):
    c = dict(n_layers=2, hidden=64, n_q_heads=4, n_kv_heads=2, head_dim=16, ffn_dim=96,
             vocab=50, rms_eps=1e-5, rope_theta=10000.0, tie_embeddings=int(tie))
    w = exact_fp8_model(c, tie)
    for mats in [w["layers"][0]["wq"], w["layers"][1]["w_down"], w["embed"]]:
        Q, s = oracle.quantize_rows(mats)   # the premise: the FP8 form is exact
        deq = np.vectorize(oracle.e4m3_to_double)(Q) * s[:, None].astype(np.float64)
        assert np.array_equal(deq, synth.bf16_to_f32(mats).astype(np.float64))
    B, mctx = 2, 24
    kc = synth.f32_to_bf16(rng.normal(0, 1, (2, B, 2, mctx, 16)).astype(np.float32))
    vc = synth.f32_to_bf16(rng.normal(0, 1, (2, B, 2, mctx, 16)).astype(np.float32))
    ref = oracle.Model(c, w, B, mctx, kc, vc)
    q8 = oracle.Model(c, w, B, mctx, kc, vc, fp8=True)
    for step in range(3):
        toks = np.array([3 + step, 40 - step], np.int32)
        pos = np.array([6 + step, 13 + step], np.int32)
        assert np.array_equal(q8.step(toks, pos), ref.step(toks, pos))
    assert np.array_equal(q8.k, ref.k) and np.array_equal(q8.v, ref.v)


def test_fp8_decode_step_differs_from_bf16_by_the_quantisation_only():
    # random weights, whose FP8 form is inexact: the FP8 step moves the
    # logits, by about the weights' relative quantisation error (<= 2^-4)
    c = dict(n_layers=1, hidden=64, n_q_heads=4, n_kv_heads=2, head_dim=16, ffn_dim=96,
             vocab=50, rms_eps=1e-5, rope_theta=10000.0, tie_embeddings=0)
    from synth.workloads import shapes
    w = {"embed": synth.f32_to_bf16(rng.normal(0, 0.2, (50, 64)).astype(np.float32)),
         "final_norm": synth.f32_to_bf16(np.ones(64, np.float32)),
         "lm_head": synth.f32_to_bf16(rng.normal(0, 0.2, (50, 64)).astype(np.float32)),
         "layers": [{k: synth.f32_to_bf16((np.ones(s) if k.endswith("norm")
                                            else rng.normal(0, 0.2, s)).astype(np.float32))
                     for k, s in shapes(c).items()}]}
    kc = synth.f32_to_bf16(rng.normal(0, 1, (1, 1, 2, 16, 16)).astype(np.float32))
    vc = kc.copy()
    a = oracle.Model(c, w, 1, 16, kc, vc).step(np.array([5], np.int32), np.array([4], np.int32))
    b = oracle.Model(c, w, 1, 16, kc, vc, fp8=True).step(np.array([5], np.int32),
                                                           np.array([4], np.int32))
    rel = np.linalg.norm(a - b) / np.linalg.norm(a)
    assert 0 < rel < 0.15
