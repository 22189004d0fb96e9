"""CPU tests of the C ABI: the library loads and exports every symbol that
include/mk.h declares; host-only planning of every workload replays cleanly
against the oracle's independent replay (bit-exact counter increments,
hazards, coverage, deadlock search); tables are deterministic; host-side
errors come back as codes with nothing launched."""
import ctypes
import os
import re

import numpy as np
import pytest

import oracle
from persistent_megakernel_decode_block_gb300 import mk
from synth.workloads import ORDER, WORKLOADS, max_ctx

HEADER = os.path.join(os.path.dirname(os.path.dirname(__file__)), "include", "mk.h")


def declared_symbols():
    text = open(HEADER).read()
    return sorted(set(re.findall(r"MK_API\s+[\w\s\*]+?\b(mk_\w+)\s*\(", text)))


def test_library_exports_every_declared_symbol():
    names = declared_symbols()
    assert len(names) >= 17
    L = ctypes.CDLL(mk.LIB)
    for n in names:
        assert hasattr(L, n), n


def host_plan(name, n_sms=152, **kw):
    w = WORKLOADS[name]
    cfg = mk.make_config(w["model"], w["batch"], max_ctx(name), num_sms=n_sms,
                         flags=mk.MK_FLAG_HOST_ONLY | kw.pop("flags", 0), **kw)
    return mk.mk_plan(cfg)


@pytest.mark.parametrize("name", ORDER)
def test_plan_replays_against_the_oracle(name):
    w = WORKLOADS[name]
    p = host_plan(name)
    try:
        info = mk.mk_plan_info(p)
        rec, raw, inc = mk.mk_plan_tables(p)
        off, idx = mk.mk_plan_lists(p)
        want = oracle.replay(raw, info["n_instr"], info["n_counters"], w["model"], w["batch"],
                             info["n_blocks"], off, idx)
        assert np.array_equal(inc, want)
        # weights are streamed exactly once per step
        m = w["model"]
        H, F, V, L = m["hidden"], m["ffn_dim"], m["vocab"], m["n_layers"]
        QD, KD = m["n_q_heads"] * m["head_dim"], m["n_kv_heads"] * m["head_dim"]
        per_layer = (QD + 2 * KD) * H + H * QD + 2 * F * H + H * F
        assert info["weight_bytes"] == 2 * (L * per_layer + V * H)
        # the phase table partitions the queue
        ph = mk.mk_plan_phases(p)
        assert sum(c for _, c, _, _ in ph) == info["n_instr"]
        assert all(rec["phase"][f:f + c].tolist() == [i] * c for i, (f, c, _, _) in enumerate(ph))
    finally:
        mk.mk_destroy(p)


@pytest.mark.parametrize("name", ["tiny", "llama1b_ctx1024", "llama1b_b8_ragged"])
@pytest.mark.parametrize("mode", [mk.MK_SCHED_DYNAMIC, mk.MK_SCHED_STATIC])
def test_plan_never_deadlocks_in_simulation(name, mode):
    p = host_plan(name, n_sms=40, sched_mode=mode)
    try:
        info = mk.mk_plan_info(p)
        _, raw, _ = mk.mk_plan_tables(p)
        lists = mk.mk_plan_lists(p) if mode == mk.MK_SCHED_STATIC else (None, None)
        oracle.simulate(raw, info["n_instr"], info["n_counters"], info["n_blocks"],
                        info["fifo_depth"], seed=11, trials=3, list_off=lists[0],
                        list_idx=lists[1])
    finally:
        mk.mk_destroy(p)


def test_tiny_plan_exhaustive_two_sm_search():
    # every interleaving of two SMs with FIFO depth 1 finishes (tiny plan)
    w = WORKLOADS["tiny"]
    cfg = mk.make_config(w["model"], 1, 128, num_sms=2, flags=mk.MK_FLAG_HOST_ONLY)
    p = mk.mk_plan(cfg)
    try:
        info = mk.mk_plan_info(p)
        _, raw, _ = mk.mk_plan_tables(p)
        assert oracle.explore(raw, info["n_instr"], info["n_counters"], 1) > info["n_instr"]
    finally:
        mk.mk_destroy(p)


def test_tables_are_deterministic():
    a, b = host_plan("llama1b_b8_ragged"), host_plan("llama1b_b8_ragged")
    try:
        assert np.array_equal(mk.mk_plan_tables(a)[1], mk.mk_plan_tables(b)[1])
        assert np.array_equal(mk.mk_plan_tables(a)[2], mk.mk_plan_tables(b)[2])
    finally:
        mk.mk_destroy(a)
        mk.mk_destroy(b)


@pytest.mark.parametrize("name", [n for n in ORDER if WORKLOADS[n]["batch"] > 1])
def test_tensor_core_tiles_split_along_k_in_whole_balanced_slices(name):
    """Batch > 1 projection tiles: every tile names its slice (chunk < nchunk,
    nchunk >= 1, also when unsplit), a split block has slices 0..S-1 sharing
    one arrival counter, with page counts that differ by at most one."""
    p = host_plan(name)
    try:
        rec, _, _ = mk.mk_plan_tables(p)
        proj = rec[rec["op"] != mk.MK_OP_ATTN]
        proj = proj[(proj["op"] >= mk.MK_OP_QKV) & (proj["op"] <= mk.MK_OP_LMHEAD)]
        assert len(proj)
        assert (proj["nchunk"] >= 1).all() and (proj["chunk"] < proj["nchunk"]).all()
        unsplit = proj["sig2_ctr"] == mk.MK_NO_COUNTER
        assert (proj["nchunk"][unsplit] == 1).all()
        split = proj[~unsplit]
        for ctr in np.unique(split["sig_ctr"]):
            blk = split[split["sig_ctr"] == ctr]
            S = int(blk["nchunk"][0])
            assert sorted(blk["chunk"].tolist()) == list(range(S))
            assert (blk["sig2_after"] == S).all() and len(np.unique(blk["sig2_ctr"])) == 1
            assert blk["npages"].max() - blk["npages"].min() <= 1
    finally:
        mk.mk_destroy(p)


@pytest.mark.parametrize("name", [n for n in ORDER if WORKLOADS[n]["batch"] > 1])
def test_attention_records_allow_the_run_time_redeal(name):
    """Batch > 1: the kernel re-deals a layer's attention slots at run time
    (static lists) by rewriting a record's chunk, sequence and group and shifting its
    two counters: that needs the phase in (chunk, sequence, group) order and
    the counters affine in sequence and group within a layer."""
    w = WORKLOADS[name]
    B, G = w["batch"], w["model"]["n_kv_heads"]
    p = host_plan(name)
    try:
        rec, _, _ = mk.mk_plan_tables(p)
        idx = np.nonzero(rec["op"] == mk.MK_OP_ATTN)[0]
        for l in np.unique(rec["layer"][idx]):
            ii = idx[rec["layer"][idx] == l]
            assert np.array_equal(ii, np.arange(ii[0], ii[0] + len(ii)))  # contiguous
            r = rec[ii]
            j = (r["chunk"].astype(np.int64) * B + r["b"]) * G + r["g"]
            assert np.array_equal(j, np.arange(len(ii)))  # (chunk, sequence, group) order
            assert len(np.unique(r["wait_ctr"].astype(np.int64) - r["g"])) == 1
            assert len(np.unique(r["sig_ctr"].astype(np.int64) - (r["b"].astype(np.int64) * G + r["g"]))) == 1
            assert len(np.unique(r["sig2_ctr"])) == 1 and len(np.unique(r["wait_tgt"])) == 1
    finally:
        mk.mk_destroy(p)


@pytest.mark.parametrize("name", [n for n in ORDER if WORKLOADS[n]["batch"] > 1])
def test_redealt_schedule_is_a_partition_and_never_deadlocks(name):
    """The schedule the batched kernel executes from static lists, once the
    oracle re-deals each attention phase for the step's positions, is still a
    partition of the queue and completes under the oracle's simulation, for
    ragged positions that include 0 and max_ctx - 1."""
    w = WORKLOADS[name]
    B, mctx = w["batch"], max_ctx(name)
    p = host_plan(name, n_sms=40, sched_mode=mk.MK_SCHED_STATIC)
    try:
        info = mk.mk_plan_info(p)
        _, raw, _ = mk.mk_plan_tables(p)
        off, idx = mk.mk_plan_lists(p)
        rng = np.random.default_rng(5)
        for trial in range(4):
            pos = rng.integers(0, mctx, B).astype(np.int32)
            pos[0], pos[-1] = 0, mctx - 1
            ex = oracle.redeal(raw, info["n_instr"], w["model"], B, info["attn_chunk"], pos, idx)
            assert np.array_equal(np.sort(ex), np.arange(info["n_instr"]))
            oracle.simulate(raw, info["n_instr"], info["n_counters"], info["n_blocks"],
                            info["fifo_depth"], seed=trial, trials=2, list_off=off,
                            list_idx=ex)
    finally:
        mk.mk_destroy(p)


@pytest.mark.parametrize("name", ["tiny", "llama1b_ctx1024", "llama1b_b8_ragged"])
def test_hybrid_lists_cover_the_queue_and_never_deadlock(name):
    """Hybrid schedule: every projection and LM-head instruction in exactly
    one list, in queue order; one attention marker per layer in every list,
    in layer order; the oracle's simulation of the lists with per-layer
    attention queues completes."""
    w = WORKLOADS[name]
    p = host_plan(name, n_sms=40, sched_mode=mk.MK_SCHED_HYBRID)
    try:
        info = mk.mk_plan_info(p)
        rec, raw, _ = mk.mk_plan_tables(p)
        off, idx = mk.mk_plan_lists(p)
        L = w["model"]["n_layers"]
        is_mark = (idx & mk.MK_LIST_ATTN) != 0
        plain = idx[~is_mark]
        want = np.nonzero(rec["op"] != mk.MK_OP_ATTN)[0]
        assert np.array_equal(np.sort(plain), want)
        for s_ in range(len(off) - 1):
            li = idx[off[s_]:off[s_ + 1]]
            m = (li & mk.MK_LIST_ATTN) != 0
            assert np.array_equal(li[m] & ~np.uint32(mk.MK_LIST_ATTN), np.arange(L))
            assert np.all(np.diff(li[~m].astype(np.int64)) > 0)
        ph = mk.mk_plan_phases(p)
        first = np.array([f for f, c, op, l in ph if op == mk.MK_OP_ATTN], np.uint32)
        cnt = [c for f, c, op, l in ph if op == mk.MK_OP_ATTN][0]
        oracle.simulate(raw, info["n_instr"], info["n_counters"], info["n_blocks"],
                        info["fifo_depth"], seed=5, trials=2, list_off=off, list_idx=idx,
                        att_first=first, att_count=cnt)
    finally:
        mk.mk_destroy(p)


@pytest.mark.parametrize("name", ORDER)
def test_attention_phase_order(name):
    """A layer's attention chunks are chunk-major (then sequence, then group)
    wherever the phase takes more than one round of the SMs or the plan is
    batched, group-major (then chunk) otherwise."""
    w = WORKLOADS[name]
    B, G = w["batch"], w["model"]["n_kv_heads"]
    p = host_plan(name)
    try:
        rec, _, _ = mk.mk_plan_tables(p)
        r = rec[(rec["op"] == mk.MK_OP_ATTN) & (rec["layer"] == 0)]
        C = int(r["nchunk"][0])
        chunk_major = B > 1 or len(r) > 152
        if chunk_major:
            j = (r["chunk"].astype(np.int64) * B + r["b"]) * G + r["g"]
        else:
            j = r["g"].astype(np.int64) * C + r["chunk"]
        assert np.array_equal(j, np.arange(len(r)))
    finally:
        mk.mk_destroy(p)


def test_fault_flag_makes_one_target_unreachable():
    w = WORKLOADS["tiny"]
    p = host_plan("tiny", flags=mk.MK_FLAG_FAULT_WAIT)
    try:
        info = mk.mk_plan_info(p)
        _, raw, _ = mk.mk_plan_tables(p)
        with pytest.raises(AssertionError, match="signals per step|waits for"):
            oracle.replay(raw, info["n_instr"], info["n_counters"], w["model"], 1,
                          info["n_blocks"])
    finally:
        mk.mk_destroy(p)


@pytest.mark.parametrize("field, value", [
    ("hidden", 200), ("ffn_dim", 300), ("n_q_heads", 6), ("head_dim", 96), ("batch", 0),
    ("batch", 17), ("batch", 24), ("batch", 64), ("max_ctx", 100), ("page_bytes", 1000),
    ("n_layers", 0), ("attn_chunk", 24), ("sched_mode", 3),
])
def test_invalid_configs_are_rejected(field, value):
    w = WORKLOADS["tiny"]
    cfg = mk.make_config(w["model"], 1, 128, num_sms=8, flags=mk.MK_FLAG_HOST_ONLY)
    setattr(cfg, field, value)
    with pytest.raises(mk.MkError) as e:
        mk.mk_plan(cfg)
    assert e.value.code == mk.MK_ERR_CONFIG


def test_planner_choices_for_the_larger_batch_mode_and_the_hybrid_schedule():
    w = WORKLOADS["llama1b_b32_ragged"]
    # batch 32: 16 KB pages by default; 32 KB pages would need more staging
    # threads than the compute warps have, so that plan is refused
    p = mk.mk_plan(mk.make_config(w["model"], 32, 4160, num_sms=152, flags=mk.MK_FLAG_HOST_ONLY))
    try:
        info = mk.mk_plan_info(p)
        assert info["page_bytes"] == 16384 and info["kernel"] == 1
        assert info["attn_chunk"] == 384  # grouped chunks: three 16 KB key pages
    finally:
        mk.mk_destroy(p)
    cfg = mk.make_config(w["model"], 32, 4160, num_sms=152, page_bytes=32768,
                         flags=mk.MK_FLAG_HOST_ONLY)
    with pytest.raises(mk.MkError) as e:
        mk.mk_plan(cfg)
    assert e.value.code == mk.MK_ERR_CONFIG
    # the hybrid schedule does not run the per-warp stream kernel
    t = WORKLOADS["tiny"]
    cfg = mk.make_config(t["model"], 1, 128, num_sms=8, sched_mode=mk.MK_SCHED_HYBRID,
                         flags=mk.MK_FLAG_HOST_ONLY | mk.MK_FLAG_STREAM_B1)
    with pytest.raises(mk.MkError) as e:
        mk.mk_plan(cfg)
    assert e.value.code == mk.MK_ERR_CONFIG


def test_host_only_plan_refuses_device_calls():
    p = host_plan("tiny")
    try:
        buf = np.zeros(4, np.int32)
        with pytest.raises(mk.MkError) as e:
            mk.mk_decode_step(p, buf, buf, (buf, buf), buf)
        assert e.value.code == mk.MK_ERR_STATE
        with pytest.raises(mk.MkError) as e:
            mk.mk_decode_step(p, None, buf, (buf, buf), buf)
        assert e.value.code == mk.MK_ERR_ARG
        assert mk.mk_status(p) == mk.MK_ERR_STATE
    finally:
        mk.mk_destroy(p)


def test_error_strings():
    for code in [0] + list(mk.ERRORS):
        assert mk.mk_error_string(code)
    assert mk.mk_error_string(12345) == "unknown error"


def test_record_layout_matches_header():
    # offsets documented in mk.h and restated in the oracle's replay
    names = [n for n in mk.INSTR_DTYPE.names]
    offs = [mk.INSTR_DTYPE.fields[n][1] for n in names]
    assert dict(zip(names, offs)) == {
        "op": 0, "flags": 1, "layer": 2, "b": 4, "g": 6, "wait_ctr": 8, "wait_tgt": 12,
        "sig_ctr": 16, "sig2_ctr": 20, "sig2_after": 24, "row0": 28, "nrows": 32, "chunk": 36,
        "nchunk": 40, "npages": 44, "wofs": 48, "phase": 56, "reserved": 60}


def test_binding_constants_match_the_header():
    # every MK_ constant the binding defines has the header's value
    text = open(HEADER).read()
    defs = {m.group(1): int(m.group(2), 0) for m in
            re.finditer(r"#define\s+(MK_\w+)\s+(-?(?:0x[0-9a-fA-F]+|\d+))u?\b", text)}
    names = [n for n in dir(mk) if n.startswith(("MK_FLAG_", "MK_SCHED_", "MK_OP_", "MK_LIST_"))
             and isinstance(getattr(mk, n), int)]
    assert len(names) >= 15
    for n in names:
        assert n in defs and defs[n] == getattr(mk, n), n


def test_without_a_gpu_planning_on_the_device_fails_cleanly():
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    w = WORKLOADS["tiny"]
    with pytest.raises(mk.MkError) as e:
        mk.mk_plan(mk.make_config(w["model"], 1, 128))
    assert e.value.code == mk.MK_ERR_DEVICE


@pytest.mark.parametrize("name", [n for n in ORDER if WORKLOADS[n]["batch"] == 1])
def test_fp8_weight_plans(name):
    """FP8 weights: the counter graph replays as for bf16; every weight is one
    byte plus one 4-byte scale per output row; a tile's pages hold 1-byte
    items (ipp = page / SW), followed in the arena by its row scales; the
    plan runs on its own kernel instantiation."""
    w = WORKLOADS[name]
    p = host_plan(name, flags=mk.MK_FLAG_FP8_WEIGHTS)
    b = host_plan(name)
    try:
        info, binfo = mk.mk_plan_info(p), mk.mk_plan_info(b)
        assert info["kernel"] == 3 and binfo["kernel"] == 0
        rec, raw, inc = mk.mk_plan_tables(p)
        off, idx = mk.mk_plan_lists(p)
        want = oracle.replay(raw, info["n_instr"], info["n_counters"], w["model"], w["batch"],
                             info["n_blocks"], off, idx)
        assert np.array_equal(inc, want)
        assert np.array_equal(inc, mk.mk_plan_tables(b)[2])
        m = w["model"]
        H, F, V, L = m["hidden"], m["ffn_dim"], m["vocab"], m["n_layers"]
        QD, KD = m["n_q_heads"] * m["head_dim"], m["n_kv_heads"] * m["head_dim"]
        rows = L * ((QD + 2 * KD) + H + 2 * F + H) + V
        per_layer = (QD + 2 * KD) * H + H * QD + 2 * F * H + H * F
        assert info["weight_bytes"] == L * per_layer + V * H + 4 * rows
        page = info["page_bytes"]
        brec = mk.mk_plan_tables(b)[0]
        for op, K in ((mk.MK_OP_QKV, H), (mk.MK_OP_OPROJ, QD), (mk.MK_OP_GATEUP, H),
                      (mk.MK_OP_DOWN, F), (mk.MK_OP_LMHEAD, H)):
            NS = -(-K // 1024)
            while K % (NS * 256):
                NS += 1
            ipp = page // (K // NS)
            t = rec[rec["op"] == op]
            wrows = t["nrows"].astype(np.int64) * (2 if op == mk.MK_OP_GATEUP else 1)
            assert np.array_equal(t["npages"], (wrows * NS + ipp - 1) // ipp)
            assert (t["npages"] <= brec[brec["op"] == op]["npages"]).all()
            # scales follow the pages; the next tile starts 4096-aligned
            ends = t["wofs"] + t["npages"].astype(np.uint64) * page + wrows.astype(np.uint64) * 4
            assert (t["wofs"] % 4096 == 0).all() and (ends[:-1] <= t["wofs"][1:]).all()
    finally:
        mk.mk_destroy(p)
        mk.mk_destroy(b)


@pytest.mark.parametrize("batch, flags", [(8, 0), (1, mk.MK_FLAG_STREAM_B1)])
def test_fp8_weights_rejected_outside_batch_one_ring_plans(batch, flags):
    m = WORKLOADS["tiny"]["model"]
    cfg = mk.make_config(m, batch, 128, num_sms=152,
                         flags=mk.MK_FLAG_HOST_ONLY | mk.MK_FLAG_FP8_WEIGHTS | flags)
    with pytest.raises(mk.MkError) as e:
        mk.mk_plan(cfg)
    assert e.value.code == mk.MK_ERR_CONFIG
