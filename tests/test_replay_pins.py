"""Pins of the oracle's plan replay.  A small instruction table is written by
hand here from the documented record format (not by the library's planner);
the replay must accept it, derive the per-step counter increments a reader can
count by eye, and reject each planted mistake."""
import struct

import numpy as np
import pytest

import oracle

NONE = 0xFFFFFFFF
QKV, ATTN, OPROJ, GATEUP, DOWN, LM = 1, 2, 3, 4, 5, 6
CFG = dict(n_layers=2, hidden=256, n_q_heads=4, n_kv_heads=2, head_dim=64, ffn_dim=512,
           vocab=256)


def rec(op, layer=0, b=0, g=0, wait=(NONE, 0), sig=0, sig2=NONE, sig2_after=0, row0=0,
        nrows=0, chunk=0, nchunk=0):
    return struct.pack("<BBHHHIIIIIIIIIIQII", op, 0, layer, b, g, wait[0], wait[1], sig, sig2,
                       sig2_after, row0, nrows, chunk, nchunk, 0, 0, 0, 0)


def ctr(l, name, g=0):
    """counter ids: per layer 8 counters, then lm_done = 16"""
    base = 8 * l
    return {"qkv": base + g, "arr": base + 2 + g, "attn": base + 4, "o": base + 5,
            "gu": base + 6, "d": base + 7}[name]


LM_DONE, NCTR = 16, 17


def build(mut=None):
    """Two layers, H 256, 4 q / 2 kv heads of 64, F 512, V 256, batch 1:
    QKV 2 tiles per group (128 rows), attention 2 chunks per group, O/GU/D/LM
    2 tiles each.  `mut(kind, l, k, fields)` may edit fields before packing."""
    out = []

    def add(kind, l, k, **f):
        if mut:
            mut(kind, l, k, f)
        if f is not None and f.get("drop") is None:
            out.append(f)

    for l in range(2):
        wait_x = (NONE, 0) if l == 0 else (ctr(l - 1, "d"), 2)
        for g in range(2):
            for t in range(2):
                add("qkv", l, 2 * g + t, op=QKV, layer=l, g=g, wait=wait_x, sig=ctr(l, "qkv", g),
                    row0=256 * g + 128 * t, nrows=128)
        for g in range(2):
            for c in range(2):
                add("attn", l, 2 * g + c, op=ATTN, layer=l, b=0, g=g, wait=(ctr(l, "qkv", g), 2),
                    sig=ctr(l, "arr", g), sig2=ctr(l, "attn"), sig2_after=2, chunk=c, nchunk=2)
        for t in range(2):
            add("o", l, t, op=OPROJ, layer=l, wait=(ctr(l, "attn"), 2), sig=ctr(l, "o"),
                row0=128 * t, nrows=128)
        for t in range(2):
            add("gu", l, t, op=GATEUP, layer=l, wait=(ctr(l, "o"), 2), sig=ctr(l, "gu"),
                row0=256 * t, nrows=256)
        for t in range(2):
            add("d", l, t, op=DOWN, layer=l, wait=(ctr(l, "gu"), 2), sig=ctr(l, "d"),
                row0=128 * t, nrows=128)
    for t in range(2):
        add("lm", 0, t, op=LM, layer=0, wait=(ctr(1, "d"), 2), sig=LM_DONE, row0=128 * t,
            nrows=128)
    table = b"".join(rec(**{k: v for k, v in f.items()}) for f in out)
    return np.frombuffer(table, dtype=np.uint8).copy(), len(out)


def run(table, n, lists=(None, None), S=4):
    return oracle.replay(table, n, NCTR, CFG, 1, S, *lists)


def test_hand_table_is_accepted_with_countable_increments():
    t, n = build()
    assert n == 2 * (4 + 4 + 2 + 2 + 2) + 2
    inc = run(t, n)
    want = np.zeros(NCTR, np.uint32)
    for l in range(2):
        for g in range(2):
            want[ctr(l, "qkv", g)] = 2
            want[ctr(l, "arr", g)] = 2
        want[ctr(l, "attn")] = 2  # one merge per (sequence, group)
        for name in ("o", "gu", "d"):
            want[ctr(l, name)] = 2
    want[LM_DONE] = 2
    assert np.array_equal(inc, want)


@pytest.mark.parametrize("mut, why", [
    (lambda k, l, i, f: f.update(wait=(f["wait"][0], 3)) if k == "o" else None, "waits for 3 signals"),
    (lambda k, l, i, f: f.update(nrows=127) if (k, l, i) == ("d", 0, 1) else None, "not written"),
    (lambda k, l, i, f: f.update(row0=0) if (k, l, i) == ("gu", 1, 1) else None, "written twice"),
    (lambda k, l, i, f: f.update(wait=(ctr(0, "o"), 2)) if (k, l) == ("d", 0) else None, "may start before"),
    (lambda k, l, i, f: f.update(wait=(ctr(1, "qkv", 0), 2)) if (k, l, i) == ("attn", 1, 2) else None, "may start before"),
    (lambda k, l, i, f: f.update(wait=(ctr(0, "gu"), 2)) if (k, l) == ("qkv", 1) else None, "may start before"),
    (lambda k, l, i, f: f.update(wait=(ctr(1, "attn"), 2)) if (k, l) == ("gu", 0) else None, "queued at or after"),
    (lambda k, l, i, f: f.update(sig2_after=1) if k == "attn" else None, "attention fields"),
    (lambda k, l, i, f: f.update(nchunk=3, sig2_after=3) if (k, l, i) == ("attn", 0, 0) else None, "chunk count"),
    (lambda k, l, i, f: f.update(g=1) if (k, l, i) == ("qkv", 0, 0) else None, "outside group"),
    (lambda k, l, i, f: f.update(wait=(NONE, 0)) if (k, l, i) == ("o", 0, 0) else None, "without a wait"),
    (lambda k, l, i, f: f.update(sig=ctr(0, "arr", 1)) if (k, l, i) == ("o", 0, 0) else None, "arrival counter shared"),
])
def test_planted_mistakes_are_rejected(mut, why):
    t, n = build(mut)
    with pytest.raises(AssertionError, match=why):
        run(t, n)


def test_simulation_accepts_valid_and_finds_deadlock():
    t, n = build()
    for S, D in [(1, 1), (2, 2), (3, 8), (16, 4)]:
        oracle.simulate(t, n, NCTR, S, D, seed=7, trials=20)
    # an unreachable target: o-proj waits for 3 merges, only 2 ever happen
    bad, n = build(lambda k, l, i, f: f.update(wait=(f["wait"][0], 3)) if k == "o" else None)
    with pytest.raises(AssertionError, match="deadlock"):
        oracle.simulate(bad, n, NCTR, 4, 2, seed=1, trials=3)


def test_exhaustive_two_sm_search():
    t, n = build()
    states = oracle.explore(t, n, NCTR, 2)
    assert states > n
    # the first QKV tile waiting on the LM-head counter can never run, and
    # everything after it depends on it: some interleaving must deadlock
    bad, n2 = build(lambda k, l, i, f: f.update(wait=(LM_DONE, 2)) if (k, l, i) == ("qkv", 0, 0) else None)
    with pytest.raises(AssertionError, match="deadlock"):
        oracle.explore(bad, n2, NCTR, 1)


def test_static_lists():
    t, n = build()
    S = 3
    lists = [[i for i in range(n) if i % S == s] for s in range(S)]
    off = np.cumsum([0] + [len(x) for x in lists]).astype(np.uint32)
    idx = np.concatenate([np.array(x, np.uint32) for x in lists])
    run(t, n, (off, idx), S=S)
    oracle.simulate(t, n, NCTR, S, 2, seed=3, trials=10, list_off=off, list_idx=idx)
    rev = idx.copy()
    rev[0], rev[1] = rev[1], rev[0]
    with pytest.raises(AssertionError, match="queue order"):
        run(t, n, (off, rev), S=S)
    short = off.copy()
    short[-1] -= 1
    with pytest.raises(AssertionError, match="cover"):
        run(t, n, (short, idx), S=S)


# ---- run-time re-deal of batched attention slots ----------------------------
# A batched table by hand: batch 2, 2 KV groups, 2 chunks of 16 positions.
# Queue: 0 QKV | 1..8 attention, chunk-major (chunk, sequence, group) | 9 O.
RB, RG, RCH = 2, 2, 16
RCFG = dict(CFG, n_layers=1)


def redeal_table(mut=None):
    out = [dict(op=QKV, layer=0, wait=(NONE, 0), sig=0, row0=0, nrows=128)]
    for c in range(2):
        for b in range(RB):
            for g in range(RG):
                f = dict(op=ATTN, layer=0, b=b, g=g, wait=(10 + g, 2), sig=100 + b * RG + g,
                         sig2=50, sig2_after=2, chunk=c, nchunk=2)
                if mut:
                    mut(c, b, g, f)
                out.append(f)
    out.append(dict(op=OPROJ, layer=0, wait=(50, RB * RG), sig=60, row0=0, nrows=128))
    t = b"".join(rec(**f) for f in out)
    return np.frombuffer(t, dtype=np.uint8).copy(), len(out)


@pytest.mark.parametrize("pos, want", [
    # every chunk of sequence 0 has work, sequence 1 only its first: as queued
    ((20, 5), [0, 1, 2, 3, 4, 5, 6, 7, 8, 9]),
    # sequence 0 ends in chunk 0, sequence 1 reaches chunk 1: its chunk-1
    # slots move ahead of sequence 0's empty ones
    ((5, 20), [0, 1, 2, 3, 4, 7, 8, 5, 6, 9]),
    # the boundary: position 15 is the last of chunk 0, 16 the first of chunk 1
    ((15, 16), [0, 1, 2, 3, 4, 7, 8, 5, 6, 9]),
    ((16, 15), [0, 1, 2, 3, 4, 5, 6, 7, 8, 9]),
    # position 0: only the new key, in chunk 0
    ((0, 0), [0, 1, 2, 3, 4, 5, 6, 7, 8, 9]),
    ((0, 31), [0, 1, 2, 3, 4, 7, 8, 5, 6, 9]),
])
def test_redeal_lists_chunks_with_work_first(pos, want):
    t, n = redeal_table()
    assert oracle.redeal(t, n, RCFG, RB, RCH, pos).tolist() == want


def test_redeal_maps_list_slots_and_keeps_each_list_in_its_phases():
    t, n = redeal_table()
    idx = np.array([0, 2, 4, 6, 8, 1, 3, 5, 7, 9], np.uint32)  # two lists of five
    got = oracle.redeal(t, n, RCFG, RB, RCH, (5, 20), idx)
    assert got.tolist() == [0, 2, 4, 8, 6, 1, 3, 7, 5, 9]


@pytest.mark.parametrize("what", ["sig_swap", "wait_shared", "sig2", "group_major", "missing"])
def test_redeal_rejects_tables_that_do_not_allow_it(what):
    def mut(c, b, g, f):
        if what == "sig_swap" and c == 1 and b == 0:   # arrival counters of two groups swapped
            f["sig"] = 100 + b * RG + (1 - g)
        if what == "wait_shared" and g == 1:           # every group waits on group 0's counter
            f["wait"] = (10, 2)
        if what == "sig2" and c == 1 and b == 1 and g == 1:
            f["sig2"] = 51
        if what == "group_major":                      # (group, sequence, chunk) order
            f["chunk"], f["g"] = g, c
    if what == "missing":
        t, n = redeal_table()
        t = np.concatenate([t[:64 * 8], t[64 * 9:]])  # drop the last attention record
        n -= 1
    else:
        t, n = redeal_table(mut)
    with pytest.raises(AssertionError):
        oracle.redeal(t, n, RCFG, RB, RCH, (5, 20))


def test_redeal_rejects_a_list_that_repeats_a_slot():
    t, n = redeal_table()
    idx = np.array([0, 1, 2, 3, 4, 5, 6, 7, 7, 9], np.uint32)
    with pytest.raises(AssertionError):
        oracle.redeal(t, n, RCFG, RB, RCH, (5, 20), idx)


# ---- hybrid lists: projections dealt round-robin, attention claimed from a
# per-layer queue (a list entry MARK | l hands over to layer l's queue)
MARK = 0x80000000
ATT_FIRST = [4, 18]  # the hand table: 14 records per layer, attention at 4..7


def hybrid_lists(n_sms=2, drop_marker=False, bad_layer=False, repeat=False):
    t, n = build()
    rec = np.frombuffer(t.tobytes(), dtype=np.uint8).reshape(n, 64)
    lists = [[] for _ in range(n_sms)]
    k = 0
    for i in range(n):
        if rec[i, 0] == ATTN:
            l = int(rec[i, 2])
            if i == ATT_FIRST[l]:
                for s, li in enumerate(lists):
                    if not (drop_marker and l == 1):
                        li.append(MARK | (5 if bad_layer and s == 0 else l))
            continue
        lists[k % n_sms].append(i)
        k += 1
    if repeat:
        lists[0].append(lists[1][0])
    off = np.cumsum([0] + [len(li) for li in lists]).astype(np.uint32)
    idx = np.array([x for li in lists for x in li], np.uint32)
    return t, n, off, idx


def test_hybrid_lists_complete_in_simulation():
    t, n, off, idx = hybrid_lists()
    oracle.simulate(t, n, NCTR, 2, 3, seed=3, trials=20, list_off=off, list_idx=idx,
                    att_first=ATT_FIRST, att_count=4)


@pytest.mark.parametrize("kw", [dict(drop_marker=True), dict(bad_layer=True), dict(repeat=True)])
def test_hybrid_simulation_rejects_broken_lists(kw):
    t, n, off, idx = hybrid_lists(**kw)
    with pytest.raises(AssertionError):
        oracle.simulate(t, n, NCTR, 2, 3, seed=3, trials=20, list_off=off, list_idx=idx,
                        att_first=ATT_FIRST, att_count=4)
