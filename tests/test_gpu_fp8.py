"""GPU parity of the FP8-weight plans (MK_FLAG_FP8_WEIGHTS): every projection
and the LM head streamed as E4M3 codes with one scale per output row, checked
teacher-forced against the oracle running the same FP8 form of the weights
(its quantiser is pinned in test_fp8_pins.py), with the bf16 tolerances;
counters against the plan replay; the multi-kernel path bit-identical to the
megakernel."""
import numpy as np
import pytest
import torch

from persistent_megakernel_decode_block_gb300 import mk
from synth.workloads import first_tokens

from harness import Setup, kv_matches_oracle, teacher_forced

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def need_gpu():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")


def check_counters(s, n_mega, n_multi=0):
    ctr, queue, exe, epoch = mk.mk_read_counters(s.plan)
    want_ctr, want_q, want_exec, want_epoch = s.expected_counters(n_mega, n_multi)
    assert epoch == want_epoch and queue == want_q
    assert np.array_equal(ctr, want_ctr) and np.array_equal(exe, want_exec)


@pytest.mark.parametrize("sched", [mk.MK_SCHED_DYNAMIC, mk.MK_SCHED_STATIC])
@pytest.mark.parametrize("tie", [False, True])
def test_fp8_tiny_all_steps(sched, tie):
    s = Setup("tiny", sched=sched, tie=tie, fp8=True)
    try:
        assert mk.mk_plan_info(s.plan)["kernel"] == 3
        worst = teacher_forced(s, s.steps)
        print("fp8 tiny: worst max|d|=%.3g relL2=%.3g" % worst)
        check_counters(s, s.steps)
        kv_matches_oracle(s)
    finally:
        s.close()


@pytest.mark.parametrize("name, steps", [("llama1b_ctx1024", 8), ("llama1b_ctx8192", 2),
                                         ("llama8b_ctx2048", 2)])
def test_fp8_full_size(name, steps):
    s = Setup(name, sched=mk.MK_SCHED_STATIC, steps=steps, fp8=True)
    try:
        worst = teacher_forced(s, steps)
        print("fp8 %s: %d steps, worst max|d|=%.3g relL2=%.3g" % (name, steps, *worst))
        check_counters(s, steps)
        kv_matches_oracle(s)
    finally:
        s.close()


def test_fp8_multikernel_matches_megakernel():
    s = Setup("tiny", sched=mk.MK_SCHED_STATIC, with_oracle=False, fp8=True)
    try:
        tok = first_tokens(s.m, s.B, 0)
        pos = s.ctx.copy()
        kc0, vc0 = s.kc.clone(), s.vc.clone()
        a = s.gpu_step(tok, pos, "mega")
        s.kc.copy_(kc0)
        s.vc.copy_(vc0)
        b = s.gpu_step(tok, pos, "multi")
        assert np.array_equal(a, b)
    finally:
        s.close()
