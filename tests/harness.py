"""Shared set-up of the GPU tests: a seeded synthetic model uploaded to the
device through torch (memory only), a plan of the CUDA library, and the
oracle holding its own copy of the same weights and KV cache."""
import numpy as np
import torch

import oracle
import synth
from persistent_megakernel_decode_block_gb300 import mk
from synth.workloads import WORKLOADS, contexts, first_tokens, make_kv, make_model, max_ctx

# logits tolerance (per step, per sequence): max |diff| and relative L2
ATOL, RTOL_L2 = 2e-2, 1e-2


def to_dev(a):
    """numpy uint16 bf16 bits -> device int16 tensor with the same bits"""
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).cuda()


class Setup:
    def __init__(self, name, seed=0, steps=None, sched=mk.MK_SCHED_DYNAMIC, flags=0, tie=None,
                 with_oracle=True, timeout_us=0, ctx=None, mctx=None, fp8=False, **plan_kw):
        """fp8: the plan streams FP8 weights (MK_FLAG_FP8_WEIGHTS) and the
        oracle runs the same FP8 form of the weights."""
        w = WORKLOADS[name]
        self.name, self.seed, self.sched = name, seed, sched
        self.m = dict(w["model"])
        if tie is not None:
            self.m["tie_embeddings"] = int(tie)
        self.B = w["batch"]
        self.steps = w["steps"] if steps is None else steps
        # prefilled lengths (the first step's positions) and the KV capacity:
        # the workload's unless a test places the positions itself
        self.ctx = contexts(name, seed) if ctx is None else np.asarray(ctx, np.int32)
        self.mctx = max_ctx(name, seed, self.steps) if mctx is None else int(mctx)
        self.weights = make_model(self.m, seed)
        self.k0, self.v0 = make_kv(self.m, self.B, self.mctx, self.ctx, seed)
        self.oracle = (oracle.Model(self.m, self.weights, self.B, self.mctx, self.k0, self.v0,
                                    fp8=fp8) if with_oracle else None)
        if fp8:
            flags |= mk.MK_FLAG_FP8_WEIGHTS
        dev = {"embed": to_dev(self.weights["embed"]),
               "final_norm": to_dev(self.weights["final_norm"]),
               "lm_head": None if self.m["tie_embeddings"] else to_dev(self.weights["lm_head"]),
               "layers": [{k: to_dev(v) for k, v in lw.items()} for lw in self.weights["layers"]]}
        cfg = mk.make_config(self.m, self.B, self.mctx, sched_mode=sched, flags=flags,
                             wait_timeout_us=timeout_us, **plan_kw)
        self.plan = mk.mk_plan(cfg)
        self.info = mk.mk_plan_info(self.plan)
        mk.mk_load_weights(self.plan, dev)
        del dev
        self.kc, self.vc = to_dev(self.k0), to_dev(self.v0)
        self.tokens = torch.zeros(self.B, dtype=torch.int32, device="cuda")
        self.positions = torch.zeros(self.B, dtype=torch.int32, device="cuda")
        self.logits = torch.zeros(self.B, self.m["vocab"], dtype=torch.float32, device="cuda")

    def close(self):
        if self.plan is not None:
            mk.mk_destroy(self.plan)
            self.plan = None

    def gpu_step(self, tokens, positions, kind="mega", use_graph=False):
        self.tokens.copy_(torch.from_numpy(np.asarray(tokens, np.int32)))
        self.positions.copy_(torch.from_numpy(np.asarray(positions, np.int32)))
        if kind == "mega":
            mk.mk_decode_step(self.plan, self.tokens, self.positions, (self.kc, self.vc),
                              self.logits)
        else:
            mk.mk_multikernel_step(self.plan, self.tokens, self.positions, (self.kc, self.vc),
                                   self.logits, use_graph=use_graph)
        code = mk.mk_status(self.plan)
        assert code == 0, mk.mk_error_string(code)
        return self.logits.double().cpu().numpy()

    def expected_counters(self, n_mega, n_multi=0):
        """Counters, queue, exec counts and epoch the oracle's replay predicts."""
        _, raw, _ = mk.mk_plan_tables(self.plan)
        inc = oracle.replay(raw, self.info["n_instr"], self.info["n_counters"], self.m, self.B,
                            self.info["n_blocks"])
        e = n_mega + n_multi
        ctr = (inc.astype(np.uint64) * e % 2 ** 32).astype(np.uint32)
        # the global work queue is only claimed in dynamic mode: N claims plus
        # one past-the-end claim per block and step (hybrid plans claim from
        # per-layer attention queues instead)
        queue = 0 if self.sched != mk.MK_SCHED_DYNAMIC else (
            n_mega * (self.info["n_instr"] + self.info["n_blocks"])) % 2 ** 32
        return ctr, queue, np.full(self.info["n_instr"], e, np.uint32), e


def compare(gpu, ref):
    """(max |diff|, relative L2) of one sequence's logits"""
    d = gpu - ref
    return float(np.abs(d).max()), float(np.linalg.norm(d) / np.linalg.norm(ref))


def teacher_forced(setup, steps, kind="mega", use_graph=False, on_step=None):
    """Run `steps` steps; the oracle's argmax (ties -> lowest index) feeds the
    next step on both sides.  Returns the worst (max |diff|, rel L2)."""
    tok = first_tokens(setup.m, setup.B, setup.seed)
    pos = setup.ctx.copy()
    worst = (0.0, 0.0)
    for s in range(steps):
        g = setup.gpu_step(tok, pos, kind, use_graph)
        r = setup.oracle.step(tok, pos)
        for b in range(setup.B):
            a, l2 = compare(g[b], r[b])
            assert a <= ATOL and l2 <= RTOL_L2, (
                "%s step %d seq %d: max|d|=%.3g relL2=%.3g" % (setup.name, s, b, a, l2))
            worst = (max(worst[0], a), max(worst[1], l2))
        if on_step:
            on_step(s, g, r)
        tok = np.array([oracle.argmax(r[b]) for b in range(setup.B)], np.int32)
        pos = pos + 1
    return worst


def kv_matches_oracle(setup):
    """GPU KV cache vs the oracle's.  Below the prefill: identical.  Rows the
    steps wrote in layer 0: within one bf16 rounding step (both sides start
    from the same embedding row; each rounds its own value).  Rows written in
    deeper layers also carry the rounding of every earlier bf16 cache write,
    undiluted where attention has one key (position 0: the attention output
    is that key's value row), so they are held, per row of d values, to the
    tolerances of the logits: max |diff| <= ATOL and relative L2 <= RTOL_L2."""
    kg = setup.kc.cpu().numpy().view(np.uint16)
    vg = setup.vc.cpu().numpy().view(np.uint16)
    for gpu, ref in ((kg, setup.oracle.k), (vg, setup.oracle.v)):
        if np.array_equal(gpu, ref):
            continue
        a = synth.bf16_to_f32(gpu).astype(np.float64)
        b = synth.bf16_to_f32(ref).astype(np.float64)
        # layer 0: one rounding step
        bad = np.abs(a[0] - b[0]) > 2.0 ** -7 * np.maximum(np.abs(b[0]), 2.0 ** -6)
        idx = np.argwhere(bad)[:5]
        assert not bad.any(), "layer-0 KV cache differs beyond one rounding step at %s: gpu %s oracle %s" % (
            idx, a[0][tuple(idx.T)], b[0][tuple(idx.T)])
        # deeper layers: per written row
        d = a[1:] - b[1:]
        rows = np.argwhere(np.abs(d).max(axis=-1) > 0)
        for r in rows:
            dr, br = d[tuple(r)], b[1:][tuple(r)]
            l2 = np.linalg.norm(dr) / max(np.linalg.norm(br), 1e-30)
            assert np.abs(dr).max() <= ATOL and l2 <= RTOL_L2, (
                "KV row (layer %d, seq %d, group %d, pos %d): max|d|=%.3g relL2=%.3g" % (
                    r[0] + 1, r[1], r[2], r[3], np.abs(dr).max(), l2))
    return True
