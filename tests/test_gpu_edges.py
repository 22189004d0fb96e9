"""GPU parity at the edges of the KV cache and of the attention tiling.

Teacher-forced windows placed by hand (same tolerances as the workload
tests, the oracle's argmax feeding both sides):
  * position 0: the step attends to its own key and nothing else (a chunk
    with no cached rows);
  * position max_ctx - 1: the last row and the last chunk of the cache,
    including a last chunk shorter than the others;
  * windows that cross an attention-chunk boundary (64 positions) and a
    key-page boundary (256 keys of head_dim 64 fill one 32 KB page; with
    256-position chunks a chunk is one page),
at batch 1 (shared page ring; the opt-in per-warp stream kernel where it
plans the same chunks) and at batch > 1 (tensor-core kernel, dynamic queue,
static lists and the hybrid schedule).  Counters, queue and execution counts stay bit-exact
against the oracle's replay and the KV cache the steps wrote matches the
oracle's.

The batched static-list plans re-deal each attention phase at run time; the
schedule that ran (which block executed which instruction, from the
per-instruction trace) is checked against the oracle's restatement of the
re-deal for the step's positions."""
import numpy as np
import pytest
import torch

import oracle
from persistent_megakernel_decode_block_gb300 import mk
from synth.workloads import first_tokens

from harness import Setup, kv_matches_oracle, teacher_forced

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def need_gpu():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")


def check_counters(s, n):
    ctr, queue, exe, epoch = mk.mk_read_counters(s.plan)
    want_ctr, want_q, want_exec, want_epoch = s.expected_counters(n)
    assert epoch == want_epoch
    assert np.array_equal(ctr, want_ctr)
    assert queue == want_q
    assert np.array_equal(exe, want_exec)


def run_window(s, steps, chunk=None):
    if chunk is not None:
        assert s.info["attn_chunk"] == chunk, s.info["attn_chunk"]
    assert int(s.ctx.max()) + steps <= s.mctx
    worst = teacher_forced(s, steps)
    check_counters(s, steps)
    kv_matches_oracle(s)
    return worst


# (workload, first positions, max_ctx, steps, plan options, expected chunk)
B1 = {
    "pos0": ("tiny", [0], 64, 8, {}, 64),
    "last_row": ("tiny", [56], 64, 8, {}, 64),
    "short_last_chunk": ("tiny", [72], 80, 8, {}, 64),       # chunks [0,64) [64,80)
    "chunk_cross": ("tiny", [60], 192, 8, {}, 64),
    "page_cross": ("tiny", [252], 512, 8, {"attn_chunk": 256}, 256),
    "llama1b_pos0": ("llama1b_ctx1024", [0], 64, 3, {}, 64),
    "llama1b_chunk_cross": ("llama1b_ctx1024", [1021], 1088, 4, {}, 64),
    "llama1b_page_cross": ("llama1b_ctx1024", [1022], 1088, 4, {"attn_chunk": 256}, 256),
    # chunks [.., 1024) [1024, 1040): the last chunk is short, the last step
    # is at max_ctx - 1
    "llama1b_last_row": ("llama1b_ctx1024", [1036], 1040, 4, {"attn_chunk": 256}, 256),
}


# the opt-in stream kernel on every window whose chunking it plans the same
# way (it chooses its own chunk cap, so not the forced 256-position chunks)
B1_RUNS = [(c, False) for c in sorted(B1)] + [(c, True) for c in sorted(B1)
                                               if "attn_chunk" not in B1[c][4]]


@pytest.mark.parametrize("case, stream", B1_RUNS)
def test_batch1_edges(case, stream):
    name, ctx, mctx, steps, kw, chunk = B1[case]
    s = Setup(name, ctx=ctx, mctx=mctx, flags=mk.MK_FLAG_STREAM_B1 if stream else 0, **kw)
    try:
        assert s.info["kernel"] == (2 if stream else 0)
        worst = run_window(s, steps, chunk)
        print("%s%s: worst max|d|=%.3g relL2=%.3g" % (case, " stream" if stream else "", *worst))
    finally:
        s.close()


# batch > 1: tensor-core kernel.  tiny_b4_ragged, max_ctx 128 (64-position
# chunks forced): sequence 0 from position 0, 1 across the chunk boundary at
# 64, 2 up to max_ctx - 1, 3 inside chunk 0.
BATCHED = {
    "tiny_b4": ("tiny_b4_ragged", [0, 60, 120, 31], 128, 8, 64, {"attn_chunk": 64}),
    # Llama-1B batch 8, max_ctx 4096, 256-position chunks (one key page):
    # sequences from 0, across 256, 1024, 2048 and 3072, and up to 4095
    "llama1b_b8": ("llama1b_b8_ragged", [0, 255, 254, 1022, 2047, 4093, 129, 3071], 4096, 3,
                   256, {"attn_chunk": 256}),
    # the same with the planner's own chunking (384 positions: one and a half
    # key pages, so chunks straddle page boundaries at 256, 768, ...)
    "llama1b_b8_auto": ("llama1b_b8_ragged", [0, 383, 384, 767, 2047, 4093, 255, 3071], 4096,
                        3, 384, {}),
    # batch 32 (16 KB pages: 128 keys per page) with 256-position chunks, so
    # a chunk's keys and values span two pages each: sequences at 0, across
    # the page boundary inside a chunk (128), across chunk boundaries (256),
    # and up to max_ctx - 1
    "tiny_b32_2pages": ("tiny_b32_ragged",
                        [0, 126, 127, 250, 255, 380, 508, 60] * 4, 512, 4, 256,
                        {"attn_chunk": 256}),
}


@pytest.mark.parametrize("case", sorted(BATCHED))
@pytest.mark.parametrize("sched", [mk.MK_SCHED_DYNAMIC, mk.MK_SCHED_STATIC, mk.MK_SCHED_HYBRID])
def test_batched_edges(case, sched):
    name, ctx, mctx, steps, chunk, kw = BATCHED[case]
    s = Setup(name, ctx=ctx, mctx=mctx, sched=sched, **kw)
    try:
        assert s.info["kernel"] == 1
        worst = run_window(s, steps, chunk)
        print("%s: worst max|d|=%.3g relL2=%.3g" % (case, *worst))
    finally:
        s.close()


@pytest.mark.parametrize("case", sorted(BATCHED))
def test_redealt_schedule_matches_the_oracle(case):
    """Static lists, batch > 1: every instruction ran on the block whose list
    slot the oracle's re-deal gives it for the step's positions, once."""
    name, ctx, mctx, _, _, kw = BATCHED[case]
    s = Setup(name, ctx=ctx, mctx=mctx, sched=mk.MK_SCHED_STATIC, flags=mk.MK_FLAG_TRACE,
              with_oracle=False, **kw)
    try:
        _, raw, _ = mk.mk_plan_tables(s.plan)
        off, idx = mk.mk_plan_lists(s.plan)
        n = s.info["n_instr"]
        tok = first_tokens(s.m, s.B, 0)
        pos = np.asarray(ctx, np.int32)
        for step in range(2):
            s.gpu_step(tok, pos + step)
            ex = oracle.redeal(raw, n, s.m, s.B, s.info["attn_chunk"], pos + step, idx)
            owner = np.empty(n, np.int64)
            for blk in range(len(off) - 1):
                owner[ex[off[blk]:off[blk + 1]]] = blk
            tr = mk.mk_read_trace(s.plan)
            ran_on = (tr[:, 0] & 0xFFFFFFFF).astype(np.int64)
            assert np.array_equal(ran_on, owner)
            _, _, exe, _ = mk.mk_read_counters(s.plan)
            assert (exe == step + 1).all()
            # the re-deal moved some slots for these ragged positions
            assert not np.array_equal(ex, idx)
    finally:
        s.close()
