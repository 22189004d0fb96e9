// mk_plan.cpp -- the host planner.
//
// « 2 · Définition et généalogie », §2.5: the CPU builds the instruction
// list; §2.6 gives the five mechanisms this table drives: persistence (one
// block per SM), dispatch (one opcode per instruction), dependency counters
// (one wait and one signal per instruction), the paged shared-memory
// allocator (the ring and slot layout computed here) and scheduling (queue
// order, or static per-SM lists).  The "one dependency event and one trigger
// event per task" normal form and "tasks of one event at contiguous indices"
// follow the MPK paragraph of the same chapter's questions: every
// instruction has one wait counter and one signal counter, and the
// instructions of one op and layer occupy one contiguous phase of the queue.
#include "mk_plan.h"

#include <string.h>

#include <algorithm>

namespace mk {

// wb: bytes per weight (2 bf16, 1 FP8)
static void geom_for(uint32_t K, uint32_t page, uint32_t wb, OpGeom &g) {
  uint32_t NS = (K + 256 * kMaxChunks - 1) / (256 * kMaxChunks);
  while (K % (NS * 256)) NS++;
  g.K = K;
  g.NS = NS;
  g.SW = K / NS;
  g.item_bytes = wb * g.SW;
  g.ipp = page / g.item_bytes;
  g.nch = g.SW / 256;
}

static uint32_t cdiv(uint64_t a, uint64_t b) { return (uint32_t)((a + b - 1) / b); }
static uint64_t align_up(uint64_t a, uint64_t b) { return (a + b - 1) / b * b; }

int build_plan(const mk_config &cfg, uint32_t num_sms, uint32_t smem_limit, HostPlan &P,
               const char **why) {
  static const char *ok = "ok";
  *why = ok;
  const mk_config &c = cfg;
#define REJECT(msg)   \
  do {                \
    *why = msg;       \
    return MK_ERR_CONFIG; \
  } while (0)
  if (c.n_layers < 1 || c.n_layers > 4096) REJECT("n_layers must be in 1..4096");
  if (c.hidden < 256 || c.hidden % 256) REJECT("hidden must be a positive multiple of 256");
  if (c.ffn_dim < 256 || c.ffn_dim % 256) REJECT("ffn_dim must be a positive multiple of 256");
  if (c.n_kv_heads < 1 || c.n_q_heads < 1 || c.n_q_heads % c.n_kv_heads)
    REJECT("n_q_heads must be a positive multiple of n_kv_heads");
  if (c.n_q_heads / c.n_kv_heads > kMaxQpg) REJECT("at most 8 q heads per KV group");
  if (c.head_dim != 64 && c.head_dim != 128) REJECT("head_dim must be 64 or 128");
  if ((c.n_q_heads * c.head_dim) % 256) REJECT("n_q_heads*head_dim must be a multiple of 256");
  if (c.vocab < 1) REJECT("vocab must be positive");
  if (c.batch < 1 || c.batch > kMaxBatch || (c.batch > 16 && c.batch % 16))
    REJECT("batch must be in 1..16, or 32 or 48");
  if (c.max_ctx < 16 || c.max_ctx % 16) REJECT("max_ctx must be a positive multiple of 16");
  if (!(c.rms_eps >= 0.0f) || !(c.rope_theta > 0.0f)) REJECT("rms_eps >= 0 and rope_theta > 0 required");
  if (c.sched_mode != MK_SCHED_DYNAMIC && c.sched_mode != MK_SCHED_STATIC &&
      c.sched_mode != MK_SCHED_HYBRID)
    REJECT("bad sched_mode");
  if (num_sms < 1 || num_sms > 1024) REJECT("number of SMs out of range");
  // larger batches (32, 48) default to 16 KB pages: a page's B operand is then
  // batch x 64 columns, one (sequence, 8 columns) unit per staging thread
  const uint32_t page = c.page_bytes ? (uint32_t)c.page_bytes : c.batch > 16 ? 16384u : 32768u;
  if (page < 4096 || page > 65536 || page % 1024) REJECT("page_bytes must be a multiple of 1024 in 4096..65536");

  if ((c.flags & MK_FLAG_FP8_WEIGHTS) && (c.batch != 1 || (c.flags & MK_FLAG_STREAM_B1)))
    REJECT("FP8 weights: batch 1 plans on the shared page ring only");

  P = HostPlan();
  P.cfg = c;
  P.fp8 = (c.flags & MK_FLAG_FP8_WEIGHTS) != 0;
  P.num_sms = num_sms;
  P.smem_limit = smem_limit;
  P.page_bytes = page;
  const int L = c.n_layers, H = c.hidden, nq = c.n_q_heads, nkv = c.n_kv_heads, d = c.head_dim,
            F = c.ffn_dim, V = c.vocab, B = c.batch;
  const int qpg = nq / nkv, GR = (qpg + 2) * d, QD = nq * d;

  // ---- GEMV geometry and tiles -------------------------------------------
  // Each phase is cut into a multiple of the SM count of tiles whose sizes
  // differ by at most one unit, so the static round-robin lists hand every
  // block the same share of every phase (one tile per block and phase where
  // the item limit allows).  Units: rotation pairs for q/k/v rows (a pair is
  // one RoPE rotation); whole pages of rows for a tied LM head (its tiles
  // then are the plain embedding matrix); single outputs otherwise.
  const uint32_t wb = P.fp8 ? 1u : 2u;
  geom_for(H, page, wb, P.geom[MK_OP_QKV]);
  geom_for(QD, page, wb, P.geom[MK_OP_OPROJ]);
  geom_for(H, page, wb, P.geom[MK_OP_GATEUP]);
  geom_for(F, page, wb, P.geom[MK_OP_DOWN]);
  geom_for(H, page, wb, P.geom[MK_OP_LMHEAD]);
  for (int op = MK_OP_QKV; op <= MK_OP_LMHEAD; ++op) {
    if (op == MK_OP_ATTN) continue;
    const OpGeom &g = P.geom[op];
    if (g.ipp < 1 || g.nch > (uint32_t)kMaxChunks || g.NS > (uint32_t)kComputeWarps)
      REJECT("GEMV geometry does not fit the compute warps");
  }
  const uint32_t max_items = std::min<uint32_t>(kMaxItems, std::max<uint32_t>(8, kMaxItemsB / B));
  bool too_big = false;
  auto split = [&](uint32_t n_out, uint32_t unit, uint32_t step, uint32_t items_per_out) {
    const uint32_t units = cdiv(n_out, unit);
    uint32_t t = std::min(step, units);
    while (t < units && (uint64_t)cdiv(units, t) * unit * items_per_out > max_items)
      t = std::min(t + step, units);
    std::vector<uint32_t> sz(t);
    uint32_t left = n_out;
    for (uint32_t i = 0; i < t; ++i) {
      const uint32_t u = units / t + (i < units % t ? 1u : 0u);
      sz[i] = std::min(u * unit, left);
      left -= sz[i];
      if ((uint64_t)sz[i] * items_per_out > max_items) too_big = true;
    }
    return sz;
  };
  const uint32_t S_ = num_sms;
  const uint32_t lm_unit = [&] {
    const OpGeom &g = P.geom[MK_OP_LMHEAD];
    if (!c.tie_embeddings || P.fp8 || page % g.item_bytes) return 1u;
    uint32_t a = g.ipp, b2 = g.NS;
    while (b2) { const uint32_t t = a % b2; a = b2; b2 = t; }
    return g.ipp / a;  // rows per unit: a multiple of whole pages
  }();
  P.tiles[MK_OP_QKV] = split(GR, 2, std::max<uint32_t>(1, S_ / nkv), P.geom[MK_OP_QKV].NS);
  P.tiles[MK_OP_OPROJ] = split(H, 1, S_, P.geom[MK_OP_OPROJ].NS);
  P.tiles[MK_OP_GATEUP] = split(F, 1, S_, 2 * P.geom[MK_OP_GATEUP].NS);
  P.tiles[MK_OP_DOWN] = split(H, 1, S_, P.geom[MK_OP_DOWN].NS);
  P.tiles[MK_OP_LMHEAD] = split(V, lm_unit, S_, P.geom[MK_OP_LMHEAD].NS);
  if (too_big && B == 1) REJECT("a GEMV tile has too many items");
  // Batch > 1: every projection runs on the tensor cores (tcgen05, M = MR
  // weight rows, N = the batch's values and bf16 remainders).  A block of MR
  // rows is split along K into S slices of whole pages, as many as keep the
  // phase within one tile per SM; the last slice of a block to finish sums
  // the slices (in slice order) and applies the epilogue.
  P.tc = B > 1;
  // Batch 1 on request: every compute warp streams its own share of each tile
  // through a private ring of 512-byte slots (per-lane async copies) instead
  // of the shared page ring fed by the loader's bulk copies.
  P.stream = B == 1 && (c.flags & MK_FLAG_STREAM_B1);
  if (P.tc) {
    P.tc_nb = 16 * cdiv(2 * (uint32_t)B, 16);
    // accumulator columns in tensor memory: a power of two >= 32
    P.tmem_cols = 32;
    while (P.tmem_cols < P.tc_nb) P.tmem_cols *= 2;
    const uint32_t rows_of[8] = {0, (uint32_t)(nkv * GR), 0, (uint32_t)H, (uint32_t)(2 * F),
                                 (uint32_t)H, (uint32_t)V, 0};
    for (int op = MK_OP_QKV; op <= MK_OP_LMHEAD; ++op) {
      if (op == MK_OP_ATTN) continue;
      OpGeom &g = P.geom[op];
      g.MR = (op == MK_OP_QKV && GR % 128) ? 64 : 128;
      g.kc = page / (g.MR * 2);
      if (g.kc < 16 || g.kc % 16) REJECT("page too small for a tensor-core tile");
      if ((uint32_t)B * (g.kc / 8) > (kComputeWarps - 1) * 32u)
        REJECT("batch too large for the page size on the tensor-core path");
      const uint32_t blocks = cdiv(rows_of[op], g.MR);
      if (g.K % g.kc) REJECT("input width does not split into tensor-core pages");
      // as many slices as keep the phase within one tile per SM (slice s
      // takes pages [s kp / S, (s + 1) kp / S) along K)
      g.kp = g.K / g.kc;
      g.S = std::max<uint32_t>(1, std::min<uint32_t>(g.kp, num_sms / blocks));
      // outputs of each block (gate/up: MR/2 outputs = MR weight rows)
      const uint32_t per = op == MK_OP_GATEUP ? g.MR / 2 : g.MR;
      const uint32_t nout = op == MK_OP_QKV ? (uint32_t)GR : op == MK_OP_GATEUP ? (uint32_t)F
                            : op == MK_OP_LMHEAD ? (uint32_t)V : (uint32_t)H;
      P.tiles[op].clear();
      for (uint32_t r0 = 0; r0 < nout; r0 += per) P.tiles[op].push_back(std::min(per, nout - r0));
      P.gpart_floats = std::max<uint64_t>(P.gpart_floats,
                                          (uint64_t)blocks * g.S * g.MR * (uint32_t)B);
    }
  }
  auto wrows_of = [](int op, uint32_t n) { return op == MK_OP_GATEUP ? 2 * n : n; };
  auto tile_pages = [&](int op, uint32_t wrows) {
    return cdiv((uint64_t)wrows * P.geom[op].NS, P.geom[op].ipp);
  };
  // arena bytes of a batch-1 tile: its pages, then (FP8 plans) one float
  // scale per row, padded so the next tile stays 4096-aligned
  auto tile_span = [&](int op, uint32_t wrows) {
    return (uint64_t)tile_pages(op, wrows) * page +
           (P.fp8 ? align_up((uint64_t)wrows * 4, 4096) : 0);
  };
  uint32_t tile_items_max = 0;
  for (int op = MK_OP_QKV; op <= MK_OP_LMHEAD; ++op)
    for (uint32_t n : P.tiles[op])
      tile_items_max = std::max(tile_items_max, wrows_of(op, n) * P.geom[op].NS);
  // arena row k of one layer's block of an op -> byte offset of its tile
  // (relative to the block) | its row within the tile (below 4096)
  for (int op = MK_OP_QKV; op <= MK_OP_LMHEAD; ++op) {
    if (op == MK_OP_ATTN) continue;
    std::vector<uint64_t> &rt = P.rowtab[op];
    rt.clear();
    P.scaletab[op].clear();
    uint64_t toff = 0;
    const int reps = op == MK_OP_QKV ? nkv : 1;
    for (int g = 0; g < reps; ++g)
      for (uint32_t n : P.tiles[op]) {
        const uint32_t w = wrows_of(op, n);
        if (P.tc) {  // tensor-core blocks: kp pages along K; retiled by formula
          toff += (uint64_t)P.geom[op].kp * page;
          continue;
        }
        if (P.stream) {  // items in (slice, row) order: offset << 24 | rows << 12 | row
          for (uint32_t r = 0; r < w; ++r) rt.push_back((toff << 24) | ((uint64_t)w << 12) | r);
          toff += (uint64_t)w * P.geom[op].NS * P.geom[op].item_bytes;
          continue;
        }
        for (uint32_t r = 0; r < w; ++r) rt.push_back(toff | r);
        if (P.fp8)
          for (uint32_t r = 0; r < w; ++r)
            P.scaletab[op].push_back(toff + (uint64_t)tile_pages(op, w) * page + 4ull * r);
        toff += tile_span(op, w);
      }
    P.block_bytes[op] = toff;
  }

  // ---- attention chunking ----------------------------------------------
  // A chunk holds at most one page of keys and one page of values, so its
  // instruction streams two pages and indexes rows without division.
  // Automatic size: one page, halved (down to 64 positions) while the
  // attention phase would occupy fewer than half of the SMs.
  // Stream plans: a warp's keys and values of a chunk must fit its ring
  // (checked once the ring size is known); start from 128 positions at
  // d = 64 and 64 at d = 128.
  const uint32_t rpp = page / (2 * (uint32_t)d);  // key (or value) rows per page
  // Tensor-core plans with d = 64 and at most four heads per group run the
  // grouped chunk, whose keys and values may span several pages: chunks of
  // 384 positions there (28 rows per warp; measured best of 256 / 384 / 448
  // at batch 8 and 32).
  P.att_grp = P.tc && d == 64 && qpg <= 4 && (page & (page - 1)) == 0;
  const uint32_t ch_cap = P.stream ? (d == 64 ? 128u : 64u) : P.att_grp ? 384u : rpp;
  uint32_t ch = c.attn_chunk > 0 ? (uint32_t)c.attn_chunk : ch_cap;
  if (c.attn_chunk <= 0)
    while (ch > 64 && (uint64_t)B * nkv * cdiv(c.max_ctx, ch) < num_sms / 2) ch /= 2;
  if (ch % 16 || ch < 16 || (!P.stream && !P.att_grp && ch > rpp) || ch > 1024 ||
      (P.att_grp && ch > 32u * kComputeWarps))
    REJECT("attn_chunk must be a multiple of 16 and at most one page of keys");
  P.attn_chunk = ch;
  P.nchunk = cdiv(c.max_ctx, ch);
  // each compute warp keeps the scores of its share of a chunk; a head has
  // at least kComputeWarps / qpg warps.  Tensor-core plans with d = 64 and at
  // most four heads per group split a chunk's positions over all compute
  // warps instead, each warp scoring its rows for every head of the group
  // (one read of each key and value row per warp): scores [row][head].
  P.att_lmax = P.att_grp
                   ? (uint32_t)align_up((uint64_t)cdiv(ch, (uint32_t)kComputeWarps) * qpg, 4)
                   : (uint32_t)align_up(cdiv(ch, (uint32_t)(kComputeWarps / qpg)), 4);

  // ---- shared-memory layout -------------------------------------------------
  // per-slot dot products (items x batch); also the size of the storer's residual buffer
  P.res_floats = P.tc ? 4u : (uint32_t)align_up((uint64_t)tile_items_max * B, 4);
  uint32_t fixed = 0;
  auto take = [&](uint32_t bytes, uint32_t align) {
    fixed = (uint32_t)align_up(fixed, align);
    uint32_t at = fixed;
    fixed += bytes;
    return at;
  };
  // offsets are relative to the end of the ring; rebased below
  uint32_t rel_fifo = take(kFifo * 64, 64);
  uint32_t rel_meta = take(kFifo * sizeof(SlotMeta), 16);
  uint32_t rel_res = take(kFifo * P.res_floats * 4, 16);
  // attention: per-warp partials {o[d]} and {m, l}, double-buffered, then
  // per-warp scores
  uint32_t att_bytes = (2 * kComputeWarps * d + 2 * kComputeWarps * 2 + kComputeWarps * P.att_lmax) * 4;
  // grouped attention: per-warp partials {o[qpg][d]} and {m, l}[qpg], single-buffered
  if (P.att_grp)
    att_bytes = (uint32_t)(kComputeWarps * qpg * (d + 2) + kComputeWarps * P.att_lmax) * 4;
  // tensor-core plans also gather a split block's slice sums here (MR x B)
  if (P.tc) att_bytes = std::max<uint32_t>(att_bytes, 128u * (uint32_t)B * 4u);
  // Tensor-core plans whose B operand has no zero rows (2B columns exactly)
  // keep the grouped attention scratch inside the B-operand slots: those are
  // idle between projections (every MMA of a tile has completed before its
  // accumulator is read), and a projection's staging starts only after the
  // attention chunk before it has passed its last barrier.
  const bool att_in_xs = P.att_grp && P.tc_nb == 2u * (uint32_t)B;
  uint32_t rel_att = take(att_in_xs ? 0u : att_bytes, 16);
  uint32_t rel_sat = take((uint32_t)L * (nkv + 4) * 4, 16);  // the waited counters
  uint32_t rel_pos = take(2 * kMaxBatch * 4, 16);
  uint32_t rel_rope = take(B * d * 4, 16);
  uint32_t rel_normr = take(2 * kMaxBatch * 4, 16);  // double-buffered per input change
  uint32_t rel_misc = take(kMiscDescOffset + kMiscDescBytes, 16);  // flags, then the pointer table
  // the attention re-deal's per-launch tables: per chunk, the mask of the
  // sequences it has work for, and the prefix count of chunk-sequence pairs
  // with work
  uint32_t rel_deal = take(P.tc ? kMaxDealChunks * 8 + (kMaxDealChunks + 1) * 4 : 0, 16);
  uint32_t rel_rbuf = take(P.res_floats * 4, 16);  // storer's prefetched residuals
  // FP8 plans: the storer's copy of the current tile's row scales
  uint32_t wsc_floats = 0;
  if (P.fp8)
    for (int op = MK_OP_QKV; op <= MK_OP_LMHEAD; ++op)
      for (uint32_t n : P.tiles[op]) wsc_floats = std::max(wsc_floats, wrows_of(op, n));
  uint32_t rel_wsc = take(wsc_floats * 4, 16);
  // staged GEMV input (normalised x, or the attention output) and attention scores
  uint32_t xs_floats = std::max<uint32_t>(H, QD);
  if (P.tc)  // the MMA's B operand, one page's columns (kc x N bf16) per ring slot
    for (int op = MK_OP_QKV; op <= MK_OP_LMHEAD; ++op)
      if (op != MK_OP_ATTN)
        xs_floats = std::max<uint32_t>(xs_floats, kTcBufs * P.geom[op].kc * P.tc_nb / 2);
  if (att_in_xs) xs_floats = std::max<uint32_t>(xs_floats, att_bytes / 4);
  uint32_t rel_xs = take((xs_floats + kComputeWarps) * 4, 16);
  uint32_t bars_max = (2 * kMaxRing + 4 * kFifo + 4 + 2 * kTcBufs) * 8;
  uint32_t rel_bars = take(bars_max, 8);
  uint32_t avail = smem_limit > fixed + 1024 ? smem_limit - fixed - 1024 : 0;
  uint32_t ring;
  if (P.stream) {  // per-warp rings of 512-byte slots, whole commit groups
    P.ring_pages = 0;
    P.wnb = std::min<uint32_t>(kMaxWarpRing, avail / (kComputeWarps * 512u)) / kSG * kSG;
    // an item (its slots plus a partly filled group) must fit
    const uint32_t nch_max = std::max(P.geom[MK_OP_QKV].nch, std::max(P.geom[MK_OP_OPROJ].nch,
                             std::max(P.geom[MK_OP_DOWN].nch, P.geom[MK_OP_LMHEAD].nch)));
    if (P.wnb < 2 * nch_max + kSG) REJECT("shared memory too small for the per-warp rings");
    // a warp's keys and values of one attention chunk must fit its ring
    const uint32_t nqs_min = (uint32_t)(kComputeWarps - qpg) / (uint32_t)qpg + 1u;
    auto fits = [&](uint32_t cpos) {
      const uint32_t rows = cdiv(cpos, nqs_min);
      const uint32_t chunks = 2u * cdiv((uint64_t)rows * d * 2u, 512u);
      return cdiv(chunks, kSG) * kSG <= P.wnb;
    };
    if (!fits(P.attn_chunk)) {
      if (c.attn_chunk > 0) REJECT("attn_chunk too large for the per-warp rings");
      while (P.attn_chunk > 16 && !fits(P.attn_chunk)) P.attn_chunk /= 2;
      if (!fits(P.attn_chunk)) REJECT("per-warp rings too small for an attention chunk");
      P.nchunk = cdiv(c.max_ctx, P.attn_chunk);
      P.att_lmax = (uint32_t)align_up(cdiv(P.attn_chunk, (uint32_t)(kComputeWarps / qpg)), 4);
    }
    ring = (uint32_t)align_up((uint64_t)kComputeWarps * P.wnb * 512u, 1024);
  } else {
    uint32_t E = std::min<uint32_t>(kMaxRing, avail / page);
    if (E < 2) REJECT("shared memory too small for a two-page ring");
    if (P.att_grp && 2 * cdiv(P.attn_chunk, rpp) > E)
      REJECT("ring too small for an attention chunk's key and value pages");
    P.ring_pages = E;
    ring = (uint32_t)align_up(E * page, 1024);
  }
  P.off_wring = 0;
  P.off_fifo = ring + rel_fifo;
  P.off_meta = ring + rel_meta;
  P.off_res = ring + rel_res;
  P.off_att = ring + (att_in_xs ? rel_xs : rel_att);
  P.off_sat = ring + rel_sat;
  P.off_pos = ring + rel_pos;
  P.off_rope = ring + rel_rope;
  P.off_normr = ring + rel_normr;
  P.off_misc = ring + rel_misc;
  P.off_deal = ring + rel_deal;
  P.off_rbuf = ring + rel_rbuf;
  P.off_wsc = ring + rel_wsc;
  P.off_xs = ring + rel_xs;
  P.off_bars = ring + rel_bars;
  P.smem_total = ring + fixed;
  if (P.smem_total > smem_limit) REJECT("shared-memory layout exceeds the limit");

  // ---- counters ----------------------------------------------------------
  P.n_wait = (uint32_t)L * (nkv + 4);
  const uint32_t arr_base = P.n_wait;
  P.lm_ctr = arr_base + (uint32_t)L * B * nkv;
  P.n_ctr = P.lm_ctr + 1;
  // split row blocks of tensor-core plans: one arrival counter each
  P.gemv_arr_base = P.n_ctr;
  if (P.tc)
    P.n_ctr += (uint32_t)L * (uint32_t)(nkv * P.tiles[MK_OP_QKV].size() + P.tiles[MK_OP_OPROJ].size() +
                                        P.tiles[MK_OP_GATEUP].size() + P.tiles[MK_OP_DOWN].size()) +
               (uint32_t)P.tiles[MK_OP_LMHEAD].size();
  uint32_t next_arr = P.gemv_arr_base;
  P.ctr_inc.assign(P.n_ctr, 0);

  // ---- weight arena: norms, embedding, then tiles in queue order ---------
  uint64_t off = 0;
  P.off_norms = off;
  off = align_up(off + (uint64_t)(2 * L + 1) * H * 2, 4096);
  {
    const OpGeom &g = P.geom[MK_OP_LMHEAD];
    // plain: every tile but the last fills whole pages, so the LM-head block
    // is the row-major embedding matrix itself
    bool plain = page % g.item_bytes == 0;
    const std::vector<uint32_t> &t = P.tiles[MK_OP_LMHEAD];
    for (size_t i = 0; i + 1 < t.size(); ++i) plain = plain && (t[i] * g.NS) % g.ipp == 0;
    P.embed_alias = c.tie_embeddings && plain && !P.tc && !P.stream && !P.fp8;
  }
  if (!P.embed_alias) {
    P.off_embed = off;
    off = align_up(off + (uint64_t)V * H * 2, 4096);
  }
  off = align_up(off, page);

  // ---- instructions --------------------------------------------------------
  auto push = [&](mk_instr in) {
    in.phase = (uint32_t)P.phases.size() - 1;
    P.instr.push_back(in);
    P.phases.back().count++;
  };
  auto new_phase = [&](uint32_t op, uint32_t layer) {
    mk_phase ph{(uint32_t)P.instr.size(), 0, op, layer};
    P.phases.push_back(ph);
  };
  auto base = [&](uint8_t op, int l) {
    mk_instr in;
    memset(&in, 0, sizeof in);
    in.op = op;
    in.layer = (uint16_t)l;
    in.wait_ctr = MK_NO_COUNTER;
    in.sig2_ctr = MK_NO_COUNTER;
    return in;
  };
  const uint32_t nO = (uint32_t)P.tiles[MK_OP_OPROJ].size();
  const uint32_t nGU = (uint32_t)P.tiles[MK_OP_GATEUP].size();
  const uint32_t nD = (uint32_t)P.tiles[MK_OP_DOWN].size();
  const uint32_t qkv_tiles_per_group = (uint32_t)P.tiles[MK_OP_QKV].size();
  P.off_qkv.resize(L);
  P.off_o.resize(L);
  P.off_gu.resize(L);
  P.off_d.resize(L);

  // one tile per entry of P.tiles[op], or, in tensor-core plans, S slices of
  // it chained through the block's arrival counter to the phase counter
  auto emit_tile = [&](uint8_t op, mk_instr in) {
    const OpGeom &g = P.geom[op];
    const uint32_t wrows = wrows_of(op, in.nrows);
    P.weight_bytes += P.fp8 ? (uint64_t)wrows * (g.K + 4) : (uint64_t)wrows * g.K * 2;
    if (P.stream) {  // items of the tile back to back, (slice, row) order
      in.npages = 0;
      in.wofs = off;
      off += (uint64_t)wrows * g.NS * g.item_bytes;
      push(in);
      P.ctr_inc[in.sig_ctr]++;
      return;
    }
    if (!P.tc) {
      in.npages = tile_pages(op, wrows);
      in.wofs = off;
      off += tile_span(op, wrows);
      push(in);
      P.ctr_inc[in.sig_ctr]++;
      return;
    }
    if (g.S == 1) {  // unsplit: the tile finishes its rows and signals the phase
      in.chunk = 0;
      in.nchunk = 1;
      in.npages = g.kp;
      in.wofs = off;
      off += (uint64_t)in.npages * page;
      push(in);
      P.ctr_inc[in.sig_ctr]++;
      return;
    }
    const uint32_t phase_ctr = in.sig_ctr, arr = next_arr++;
    for (uint32_t sl = 0; sl < g.S; ++sl) {
      mk_instr t = in;
      t.sig_ctr = arr;
      t.sig2_ctr = phase_ctr;
      t.sig2_after = g.S;
      t.chunk = sl;
      t.nchunk = g.S;
      t.npages = (sl + 1) * g.kp / g.S - sl * g.kp / g.S;
      t.wofs = off;
      off += (uint64_t)t.npages * page;
      push(t);
      P.ctr_inc[arr]++;
    }
    P.ctr_inc[phase_ctr]++;
  };
  auto gemv_tiles = [&](uint8_t op, mk_instr proto) {
    uint32_t row0 = 0;
    for (uint32_t n : P.tiles[op]) {
      mk_instr in = proto;
      in.row0 = row0;
      in.nrows = n;
      row0 += n;
      emit_tile(op, in);
    }
  };

  for (int l = 0; l < L; ++l) {
    // RMSNorm + QKV + RoPE, group-major so a group's attention can start early
    new_phase(MK_OP_QKV, l);
    P.off_qkv[l] = off;
    for (int grp = 0; grp < nkv; ++grp) {
      uint32_t r0 = 0;
      for (uint32_t n : P.tiles[MK_OP_QKV]) {
        mk_instr in = base(MK_OP_QKV, l);
        in.flags = l == 0 ? 1 : 0;
        in.g = (uint16_t)grp;
        if (l > 0) {
          in.wait_ctr = ctr_d(c, l - 1);
          in.wait_tgt = nD;
        }
        in.sig_ctr = ctr_qkv(c, l, grp);
        in.row0 = grp * GR + r0;
        in.nrows = n;
        r0 += n;
        emit_tile(MK_OP_QKV, in);
      }
    }
    // attention chunks, group-major
    new_phase(MK_OP_ATTN, l);
    // Order of the phase.  Where it takes several rounds of the SMs (and in
    // every batched plan): chunk-major, then sequence, then group, so that
    // dealt round-robin each group's chunks spread over the rounds alike and
    // every group's merge comes at about the same time; batched plans also
    // re-deal this order at run time (static lists) so that chunks with work
    // (a ragged batch's early chunks) spread evenly.  One round at batch 1:
    // group-major, a group's chunks next to each other.
    const uint32_t n_att = P.nchunk * (uint32_t)B * (uint32_t)nkv;
    const bool chunk_major = B > 1 || n_att > num_sms;
    for (uint32_t jj = 0; jj < n_att; ++jj) {
        const uint32_t ck = chunk_major ? jj / ((uint32_t)B * nkv) : jj % P.nchunk;
        const int b = chunk_major ? (int)((jj / nkv) % B) : 0;
        const int grp = chunk_major ? (int)(jj % nkv) : (int)(jj / P.nchunk);
        {
          mk_instr in = base(MK_OP_ATTN, l);
          in.b = (uint16_t)b;
          in.g = (uint16_t)grp;
          in.wait_ctr = ctr_qkv(c, l, grp);
          in.wait_tgt = qkv_tiles_per_group;
          in.sig_ctr = arr_base + ((uint32_t)l * B + b) * nkv + grp;
          in.sig2_ctr = ctr_attn(c, l);
          in.sig2_after = P.nchunk;
          in.chunk = ck;
          in.nchunk = P.nchunk;
          push(in);
          P.ctr_inc[in.sig_ctr]++;
          if (ck == 0) P.ctr_inc[in.sig2_ctr]++;
        }
    }
    // O-projection + residual
    new_phase(MK_OP_OPROJ, l);
    P.off_o[l] = off;
    {
      mk_instr in = base(MK_OP_OPROJ, l);
      in.flags = l == 0 ? 1 : 0;
      in.wait_ctr = ctr_attn(c, l);
      in.wait_tgt = (uint32_t)B * nkv;
      in.sig_ctr = ctr_o(c, l);
      gemv_tiles(MK_OP_OPROJ, in);
    }
    // RMSNorm + gate/up + SiLU*mul
    new_phase(MK_OP_GATEUP, l);
    P.off_gu[l] = off;
    {
      mk_instr in = base(MK_OP_GATEUP, l);
      in.wait_ctr = ctr_o(c, l);
      in.wait_tgt = nO;
      in.sig_ctr = ctr_gu(c, l);
      gemv_tiles(MK_OP_GATEUP, in);
    }
    // down-projection + residual
    new_phase(MK_OP_DOWN, l);
    P.off_d[l] = off;
    {
      mk_instr in = base(MK_OP_DOWN, l);
      in.wait_ctr = ctr_gu(c, l);
      in.wait_tgt = nGU;
      in.sig_ctr = ctr_d(c, l);
      gemv_tiles(MK_OP_DOWN, in);
    }
  }
  new_phase(MK_OP_LMHEAD, 0);
  P.off_lm = off;
  {
    mk_instr in = base(MK_OP_LMHEAD, 0);
    in.wait_ctr = ctr_d(c, L - 1);
    in.wait_tgt = nD;
    in.sig_ctr = P.lm_ctr;
    gemv_tiles(MK_OP_LMHEAD, in);
  }
  P.arena_bytes = align_up(off, 4096);

  // test-only fault: one wait target that can never be reached
  if (c.flags & MK_FLAG_FAULT_WAIT) {
    const mk_phase &ph = P.phases[5 * (L - 1) + 2];  // O-projection of the last layer
    P.fault_instr = ph.first;
    P.instr[ph.first].wait_tgt += 1;
  }

  // ---- static per-SM lists: round-robin over the queue order -------------
  // Hybrid: the projections (and the LM head) are dealt round-robin as in
  // static lists; each attention phase becomes one marker entry in every
  // list, where the block claims from that layer's attention queue.
  P.att_first.assign(L, 0);
  for (const mk_phase &ph : P.phases)
    if (ph.op == MK_OP_ATTN) P.att_first[ph.layer] = ph.first;
  P.att_count = P.nchunk * (uint32_t)B * (uint32_t)nkv;
  if (c.sched_mode == MK_SCHED_HYBRID) {
    if (P.stream) REJECT("the hybrid schedule does not run the per-warp stream kernel");
    std::vector<std::vector<uint32_t>> lists(num_sms);
    uint32_t k = 0;
    for (const mk_phase &ph : P.phases) {
      if (ph.op == MK_OP_ATTN) {
        for (auto &li : lists) li.push_back(MK_LIST_ATTN | ph.layer);
        continue;
      }
      for (uint32_t i = ph.first; i < ph.first + ph.count; ++i) lists[k++ % num_sms].push_back(i);
    }
    P.list_off.assign(num_sms + 1, 0);
    P.list_idx.clear();
    for (uint32_t s = 0; s < num_sms; ++s) {
      P.list_idx.insert(P.list_idx.end(), lists[s].begin(), lists[s].end());
      P.list_off[s + 1] = (uint32_t)P.list_idx.size();
    }
  } else {
    P.list_off.assign(num_sms + 1, 0);
    for (uint32_t s = 0; s < num_sms; ++s)
      P.list_off[s + 1] = P.list_off[s] + (uint32_t)((P.instr.size() + num_sms - 1 - s) / num_sms);
    P.list_idx.resize(P.instr.size());
    for (uint32_t s = 0, k = 0; s < num_sms; ++s)
      for (size_t i = s; i < P.instr.size(); i += num_sms) P.list_idx[k++] = (uint32_t)i;
  }

  // ---- re-tiling maps ----------------------------------------------------
  P.qkv_map.resize((size_t)(nq + 2 * nkv) * d);
  for (int R = 0; R < (nq + 2 * nkv) * d; ++R) {
    int grp = R / GR, q = R % GR;
    auto pair_to_natural = [&](int ip) { return ip % 2 == 0 ? ip / 2 : ip / 2 + d / 2; };
    int nat;
    if (q < qpg * d)
      nat = (grp * qpg + q / d) * d + pair_to_natural(q % d);
    else if (q < (qpg + 1) * d)
      nat = QD + grp * d + pair_to_natural(q - qpg * d);
    else
      nat = QD + nkv * d + grp * d + (q - (qpg + 1) * d);
    P.qkv_map[R] = nat;
  }
  {
    P.gu_map.resize((size_t)2 * F);
    size_t k = 0;
    uint32_t r0 = 0;
    for (uint32_t nr : P.tiles[MK_OP_GATEUP]) {
      if (P.tc) {  // tensor-core tiles interleave: row 2j gate j, row 2j + 1 up j
        for (uint32_t j = 0; j < nr; ++j) {
          P.gu_map[k++] = (int32_t)(r0 + j);
          P.gu_map[k++] = (int32_t)(F + r0 + j);
        }
      } else {  // GEMV tiles: the tile's gate rows, then its up rows
        for (uint32_t j = 0; j < nr; ++j) P.gu_map[k++] = (int32_t)(r0 + j);
        for (uint32_t j = 0; j < nr; ++j) P.gu_map[k++] = (int32_t)(F + r0 + j);
      }
      r0 += nr;
    }
  }

#undef REJECT
  return MK_OK;
}

}  // namespace mk
