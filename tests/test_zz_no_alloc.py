"""The allocation-free attention entry point (mk_attention_noalloc), for
callers that cannot allocate device memory themselves, e.g. an engine whose
GPU memory is all owned by its own allocator.  Its chunk partials live in the
library's fixed static device array.  Checked through the C ABI against the
oracle's attention (fp64, one query head at a time, on the seeded inputs) and
against the plan-based path that computes the same attention (the attention
phase of a layer, run alone with mk_run_phase), on two calls in a row, so a
second call that reuses the shared array must still be right; head_dim 128
and an out-of-range position (NaN rows) without a plan.  Kept in the file
pytest collects last."""
import numpy as np
import pytest
import torch

import oracle
import synth
from persistent_megakernel_decode_block_gb300 import mk

from harness import ATOL, RTOL_L2, Setup, compare

pytestmark = pytest.mark.gpu


class _DevView:
    """A torch view of a raw device pointer of the plan (fp32)."""

    def __init__(self, ptr, n):
        self.__cuda_array_interface__ = {"data": (ptr, False), "shape": (n,),
                                         "typestr": "<f4", "version": 3}


def _view(ptr, n):
    return torch.as_tensor(_DevView(ptr, n), device="cuda")


@pytest.mark.parametrize("name", ["tiny", "llama1b_b8_ragged"])
def test_no_alloc_attention_matches_the_plan_path(name):
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    s = Setup(name, with_oracle=False)
    try:
        m, B = s.m, s.B
        nq, nkv, d, L = m["n_q_heads"], m["n_kv_heads"], m["head_dim"], m["n_layers"]
        buf = mk.mk_debug_buffers(s.plan)
        q_plan = _view(buf["q"], B * nq * d)
        attn_plan = _view(buf["attn"], B * nq * d)
        phases = mk.mk_plan_phases(s.plan)
        gen = torch.Generator(device="cpu").manual_seed(7)
        s.positions.copy_(torch.from_numpy(s.ctx.astype(np.int32)))
        layer_elems = B * nkv * s.mctx * d
        for layer in (0, L - 1):
            ph = [i for i, (_, _, op, l) in enumerate(phases) if op == mk.MK_OP_ATTN and l == layer][0]
            q = torch.randn(B * nq * d, generator=gen).cuda()
            q_plan.copy_(q)
            mk.mk_reset(s.plan)
            mk.mk_run_phase(s.plan, ph, s.tokens, s.positions, (s.kc, s.vc), s.logits)
            assert mk.mk_status(s.plan) == 0
            ref = attn_plan.double().cpu().numpy().reshape(B, -1)
            # the oracle on the seeded inputs: q as drawn, the layer's cache as generated
            qh = q.cpu().double().numpy().reshape(B, nq, d)
            qpg = nq // nkv
            for b in range(B):
                n = int(s.ctx[b]) + 1
                want = np.concatenate([oracle.attention(qh[b, h], s.k0[layer, b, h // qpg, :n],
                                                        s.v0[layer, b, h // qpg, :n])
                                       for h in range(nq)])
                a, l2 = compare(ref[b], want)
                assert a <= ATOL and l2 <= RTOL_L2, ("plan path vs oracle", layer, b, a, l2)
            kl = s.kc.view(-1)[layer * layer_elems:]
            vl = s.vc.view(-1)[layer * layer_elems:]
            for call in range(2):  # the second call reuses the shared scratch
                out = torch.full((B, nq * d), float("nan"), device="cuda")
                mk.mk_attention_noalloc(q, kl, vl, s.positions, out, B, nq, nkv, d, s.mctx)
                torch.cuda.synchronize()
                got = out.double().cpu().numpy()
                for b in range(B):
                    a, l2 = compare(got[b], ref[b])
                    assert a <= ATOL and l2 <= RTOL_L2, (layer, call, b, a, l2)
                    qh_b = q.cpu().double().numpy().reshape(B, nq, d)[b]
                    n = int(s.ctx[b]) + 1
                    want = np.concatenate([oracle.attention(qh_b[h], s.k0[layer, b, h // qpg, :n],
                                                            s.v0[layer, b, h // qpg, :n])
                                           for h in range(nq)])
                    a, l2 = compare(got[b], want)
                    assert a <= ATOL and l2 <= RTOL_L2, ("no-alloc vs oracle", layer, call, b, a, l2)
    finally:
        s.close()


def test_no_alloc_attention_rejects_what_does_not_fit():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    x = torch.zeros(16, device="cuda")
    p = torch.zeros(16, dtype=torch.int32, device="cuda")
    with pytest.raises(mk.MkError) as e:  # 16 x 8 x 512 chunks of 1040 floats > 4 MiB
        mk.mk_attention_noalloc(x, x, x, p, x, 16, 64, 8, 128, 131072)
    assert e.value.code == mk.MK_ERR_ARG
    with pytest.raises(mk.MkError) as e:
        mk.mk_attention_noalloc(x, x, x, p, x, 1, 6, 4, 64, 128)
    assert e.value.code == mk.MK_ERR_ARG


def test_no_alloc_attention_head_dim_128_and_out_of_range_rows():
    """head_dim 128 (the Llama-8B head), 2 KV groups of 4 query heads, a
    512-position cache; sequences at positions 0, 300 and 511 = max_ctx - 1
    match the oracle, a sequence at position max_ctx gets NaN rows."""
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    B, nq, nkv, d, mctx = 4, 8, 2, 128, 512
    qpg = nq // nkv
    pos = np.array([0, 300, 511, 512], np.int32)
    k = synth.normal_bf16(3, 901, (B, nkv, mctx, d))
    v = synth.normal_bf16(3, 902, (B, nkv, mctx, d))
    q = torch.randn(B * nq * d, generator=torch.Generator().manual_seed(11))
    kd = torch.from_numpy(k.view(np.int16)).cuda()
    vd = torch.from_numpy(v.view(np.int16)).cuda()
    pd = torch.from_numpy(pos).cuda()
    out = torch.zeros((B, nq * d), device="cuda")
    mk.mk_attention_noalloc(q.cuda(), kd, vd, pd, out, B, nq, nkv, d, mctx)
    torch.cuda.synchronize()
    got = out.double().cpu().numpy()
    qh = q.double().numpy().reshape(B, nq, d)
    for b in range(3):
        n = int(pos[b]) + 1
        want = np.concatenate([oracle.attention(qh[b, h], k[b, h // qpg, :n], v[b, h // qpg, :n])
                               for h in range(nq)])
        a, l2 = compare(got[b], want)
        assert a <= ATOL and l2 <= RTOL_L2, (b, a, l2)
    assert np.isnan(got[3]).all()
