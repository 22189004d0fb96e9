// mk_kernel.cu -- the persistent decode megakernel (sm_103a).
//
// One launch runs a whole decoder forward pass (« 2 · Définition et
// généalogie », §2.1).  The grid holds one resident block per SM (§2.6,
// "1. La persistance"); each block interprets instructions taken from a
// global work queue or from its own list (§2.4, persistent-threads loop;
// §2.6, "2. Le dispatch d'instructions" and "5. L'ordonnancement").  Inside
// a block the warps are specialised (« 5 · La spécialisation des warps »,
// §5.2 and §5.4):
//   warp 0       loader : claims instructions, streams their weight pages
//                (or KV-cache rows) with bulk async copies into a ring of
//                shared-memory pages tracked by full/empty mbarriers (§5.2's
//                producer/consumer ring; §2.6, "4. L'allocateur de mémoire
//                partagée"), and runs ahead across dependency waits (§5.4:
//                load the next op's weights while the current one finishes).
//   warp 1       storer : epilogues (RoPE, KV append, residual add, SiLU,
//                attention merge), global stores, then the release of the
//                instruction's dependency counter (§2.6, "3. Les compteurs").
//   warps 2..15  compute: wait on the instruction's counter (acquire), then
//                bf16 GEMV with fp32 accumulation from the ring pages, or a
//                split-KV attention chunk.
// Every wait is bounded by %globaltimer; on expiry the block latches
// MK_ERR_TIMEOUT, raises a global abort flag that every other wait polls,
// waits for its own copies in flight and returns.
#include <cuda_fp16.h>
#include <cuda_fp8.h>

#include <algorithm>

#include "mk_device.cuh"

namespace mk {


// pages the loader streams for an instruction
DEVI uint32_t n_pages(const KParams &P, const Smem &S, const mk_instr &in) {
  if (in.op != MK_OP_ATTN) return in.npages;
  int p0, p1;
  const int pos = S.pos[in.b];
  attn_range(P, pos, in.chunk, p0, p1);
  const int n_old = max(0, min(p1, pos) - p0);
  const int rpp = P.page_bytes / (P.d * 2);
  return 2u * (uint32_t)((n_old + rpp - 1) / rpp);
}

DEVI void page_src(const KParams &P, const Smem &S, const mk_instr &in, uint32_t p,
                   uint32_t np, const void *&src, uint32_t &bytes) {
  if (in.op != MK_OP_ATTN && P.tc) {  // tensor-core tiles are whole pages
    src = P.arena + in.wofs + (uint64_t)p * P.page_bytes;
    bytes = P.page_bytes;
    return;
  }
  if (in.op != MK_OP_ATTN) {
    const OpGeom &G = P.geom[in.op];
    const uint32_t wrows = in.op == MK_OP_GATEUP ? 2 * in.nrows : in.nrows;
    const uint32_t items = wrows * G.NS;
    const uint32_t n = min(G.ipp, items - p * G.ipp);
    src = P.arena + in.wofs + (uint64_t)p * P.page_bytes;
    bytes = n * G.item_bytes;
    return;
  }
  int p0, p1;
  const int pos = S.pos[in.b];
  attn_range(P, pos, in.chunk, p0, p1);
  const int n_old = max(0, min(p1, pos) - p0);
  const int rpp = P.page_bytes / (P.d * 2);
  const uint32_t npk = np / 2;
  const bool is_v = p >= npk;
  const int pp = (int)(is_v ? p - npk : p);
  const int r0 = pp * rpp, rows = min(rpp, n_old - r0);
  const uint16_t *base = (is_v ? P.vc : P.kc) + kv_row(P, in.layer, in.b, in.g, p0 + r0);
  src = base;
  bytes = (uint32_t)rows * P.d * 2;
}

// --------------------------------------------------------------- loader ----
DEVI void drain_copies(const KParams &P, const Smem &S, uint32_t seq) {
  const uint32_t E = P.ring_pages;
  const uint32_t first = seq > E ? seq - E : 0;
  for (uint32_t s = first; s < seq; ++s) {
    uint64_t *bar = &S.full[s % E];
    const uint32_t par = (s / E) & 1u;
    const uint64_t t0 = cycles();
    while (!mbar_try_wait(bar, par))
      if (cycles() - t0 > 500000000ull) {  // >= 200 ms: a bulk copy never takes that long
        raise_error(P, MK_ERR_TIMEOUT, kWhereDrain | s, true);
        break;
      }
  }
}

// The loader is one thread running two cursors over the FIFO:
//  * claim cursor: takes the next instruction (queue claim, list entry or
//    range), copies its record into a free FIFO slot with its page range and
//    publishes it -- up to P.lookahead entries ahead of the stream cursor,
//    independently of any dependency.  Claims and record loads are issued two
//    instructions ahead so a burst of publishes does not wait on them;
//  * stream cursor: copies the published pages, in order, into the
//    shared-memory ring as slots are released by the compute warps.
// Nothing here waits on a dependency counter, so the weights of later
// instructions keep flowing while the compute warps wait (pages' §5.4).
DEVI void load_record(const KParams &P, uint32_t idx, uint4 (&r)[4]) {
  if (idx < P.n_instr) {
    const uint4 *src = reinterpret_cast<const uint4 *>(P.instr + idx);
#pragma unroll
    for (int i = 0; i < 4; ++i) r[i] = __ldg(src + i);
  }
}

// Static lists and ragged batches: whether an attention chunk has work
// depends on its sequence's position, known only at run time, so a fixed
// round-robin of chunk instructions can hand one SM six chunks with work and
// another two.  Instead the list slots of a layer's attention phase are
// re-dealt at run time, identically on every SM: slot j (phase order: chunk,
// sequence, group) takes the j-th instruction of the phase in an order that
// lists every chunk with work first, so chunks with work are spread over the
// SMs like the slots.  Rewrites the FIFO copy of the record (chunk, sequence,
// group and their two counters, affine in sequence and group) and returns the
// index of the instruction it now is.
// n-th (0-based) set bit of a 64-bit mask that has more than n set bits
DEVI int nth_set_bit(uint64_t m, int n) {
  const uint32_t lo = (uint32_t)m, hi = (uint32_t)(m >> 32);
  const int nlo = __popc(lo);
  return n < nlo ? (int)__fns(lo, 0, n + 1) : 32 + (int)__fns(hi, 0, n - nlo + 1);
}

DEVI uint32_t balance_attn(const KParams &P, const Smem &S, mk_instr &in, uint32_t idx) {
  const int B = P.B, G = P.nkv, C = (int)in.nchunk, ch = P.attn_chunk;
  const int j = ((int)in.chunk * B + in.b) * G + in.g;
  if (C <= kMaxDealChunks) {
    // from the launch's tables: binary search of the chunk, the rank's
    // sequence as the n-th set bit of the chunk's mask (or of its complement)
    const int nreal = (int)S.dpre[C] * G;
    const bool want_real = j < nreal;
    const int r = want_real ? j : j - nreal;
    const int q = r / G, g = r % G;  // rank of the (chunk, sequence) pair, group
    auto before = [&](int c) {        // pairs of the wanted kind in chunks < c
      return want_real ? (int)S.dpre[c] : c * B - (int)S.dpre[c];
    };
    int lo = 0, hi = C - 1;  // last chunk c with before(c) <= q
    while (lo < hi) {
      const int mid = (lo + hi + 1) / 2;
      if (before(mid) <= q) lo = mid;
      else hi = mid - 1;
    }
    const int c = lo;
    const uint64_t all = B == 64 ? ~0ull : (1ull << B) - 1ull;
    const uint64_t m = want_real ? S.dmask[c] : (~S.dmask[c] & all);
    const int b = nth_set_bit(m, q - before(c));
    const int jn = (c * B + b) * G + g;
    in.sig_ctr = in.sig_ctr + (uint32_t)((b - (int)in.b) * G + (g - (int)in.g));
    in.wait_ctr = in.wait_ctr + (uint32_t)(g - (int)in.g);
    in.chunk = (uint32_t)c;
    in.b = (uint16_t)b;
    in.g = (uint16_t)g;
    return idx - (uint32_t)j + (uint32_t)jn;
  }
  // sequences whose position reaches chunk c: those with pos >= c * ch
  auto live = [&](int c) {
    int n = 0;
    for (int b = 0; b < B; ++b) n += S.pos[b] >= c * ch;
    return n;
  };
  int nreal = 0;
  for (int c = 0; c < C; ++c) nreal += live(c) * G;
  const bool want_real = j < nreal;
  int r = want_real ? j : j - nreal;  // rank among the chunks with (without) work
  int c = 0;
  for (; c < C; ++c) {
    const int n = (want_real ? live(c) : B - live(c)) * G;
    if (r < n) break;
    r -= n;
  }
  // the (r / G)-th sequence of chunk c with (without) work, group r % G
  int b = 0, k = r / G;
  for (; b < B; ++b)
    if ((S.pos[b] >= c * ch) == want_real && k-- == 0) break;
  const int g = r % G;
  const int jn = (c * B + b) * G + g;
  in.sig_ctr = in.sig_ctr + (uint32_t)((b - (int)in.b) * G + (g - (int)in.g));
  in.wait_ctr = in.wait_ctr + (uint32_t)(g - (int)in.g);
  in.chunk = (uint32_t)c;
  in.b = (uint16_t)b;
  in.g = (uint16_t)g;
  return idx - (uint32_t)j + (uint32_t)jn;
}

// HYB: the hybrid schedule's claims and publish gate (compiled only into the
// loader that runs hybrid plans, so the others' polling loop stays as short)
template <bool TC, bool HYB>
DEVI void loader(const KParams &P, const Smem &S, uint32_t epoch) {
  const uint64_t pol = policy_evict_first();
  const uint32_t N = P.n_instr, E = P.ring_pages, PG = P.page_bytes;
  const uint32_t qbase = epoch * (N + P.n_blocks);
  uint32_t list_k = 0, list_end = 0, range_taken = 0;
  int att_l = -1;  // hybrid: the layer whose attention queue this block claims from
  if (P.mode == kModeStatic || P.mode == kModeHybrid) {
    list_k = P.list_off[blockIdx.x];
    list_end = P.list_off[blockIdx.x + 1];
  }
  // every block takes exactly one past-the-end claim: no claim follows an
  // index >= N
  auto claim = [&]() -> uint32_t {
    if (P.mode == kModeDynamic) return atomicAdd(P.ctrl + kCtlQueue, 1u) - qbase;
    if (P.mode == kModeStatic) return list_k < list_end ? __ldg(P.list_idx + list_k++) : N;
    if (HYB) {
      // the list, where an attention marker hands over to that layer's queue
      // until it is empty (every block takes one failing claim per layer)
      while (true) {
        if (att_l >= 0) {
          const uint32_t j = atomicAdd(P.aq + att_l, 1u) - epoch * (P.att_count + P.n_blocks);
          if (j < P.att_count) return __ldg(P.att_first + att_l) + j;
          att_l = -1;
        }
        if (list_k >= list_end) return N;
        const uint32_t e = __ldg(P.list_idx + list_k++);
        if (!(e & MK_LIST_ATTN)) return e;
        att_l = (int)(e & ~MK_LIST_ATTN);
      }
    }
    const uint32_t r = range_taken ? N : P.range_first + blockIdx.x;
    range_taken = 1;
    return r;
  };
  // pipeline: a (next to publish, record ra), b (record rb), c (claim only)
  uint4 ra[4], rb[4];
  uint32_t a = claim(), b = N, c = N;
  load_record(P, a, ra);
  if (a < N) b = claim();
  load_record(P, b, rb);
  if (b < N) c = claim();
  uint32_t fs_c = 0, seq_c = 0;            // claim cursor: FIFO entry, first page of it
  uint32_t fs_s = 0, p_s = 0, seq_s = 0;   // stream cursor: FIFO entry, page in it, ring seq
  uint32_t fs_p = 0, p_p = 0, seq_p = 0;   // L2-prefetch cursor (never behind the stream)
  bool ended = false;                      // END published at entry fs_c - 1
  bool ok = true;
  uint64_t t_idle = 0;  // start of the current idle stretch (0: not idle)
  uint32_t n_idle = 0;
  while (true) {
    bool progress = false;
    // ---- claim cursor
    // hybrid: an attention chunk claimed from a queue is published only once
    // the compute warps have started the entry before it, so a block takes
    // chunks as it drains them, not as fast as its loader runs ahead
    const bool gate = HYB && a < N && (ra[0].x & 0xFFu) == MK_OP_ATTN &&
                      fs_c > 0 &&
                      !mbar_test(&S.rdy[(fs_c - 1) % kFifo], ((fs_c - 1) / kFifo) & 1u);
    if (!ended && !gate && fs_c - fs_s < P.lookahead) {
      const uint32_t f = fs_c % kFifo, k = fs_c / kFifo;
      if (k == 0 || mbar_test(&S.iempty[f], (k - 1) & 1u)) {
        if (a >= N) {
          S.fifo[f].op = MK_OP_END;
          S.meta[f].idx = N;
          S.meta[f].npages = 0;
          mbar_arrive(&S.ifull[f]);
          ended = true;
        } else {
          uint4 *dst = reinterpret_cast<uint4 *>(&S.fifo[f]);
#pragma unroll
          for (int i = 0; i < 4; ++i) dst[i] = ra[i];
          uint32_t idx = a;
          if (TC && (P.mode == kModeStatic || HYB) &&
              S.fifo[f].op == MK_OP_ATTN)  // (batch > 1)
            idx = balance_attn(P, S, S.fifo[f], a);
          const mk_instr &in = S.fifo[f];
          const uint32_t np = n_pages(P, S, in);
          SlotMeta &m = S.meta[f];
          m.idx = idx;
          m.seq0 = seq_c;
          m.npages = np;
          m.t_claim = (P.flags & MK_FLAG_TRACE) ? gtimer() : 0ull;
          mbar_arrive(&S.ifull[f]);
          seq_c += np;
          // advance the pipeline
          a = b;
#pragma unroll
          for (int i = 0; i < 4; ++i) ra[i] = rb[i];
          b = c;
          load_record(P, b, rb);
          c = b < N ? claim() : N;
        }
        ++fs_c;
        progress = true;
      }
    }
    // ---- L2-prefetch cursor: up to l2_window bytes of published pages ahead
    // of the ring, so pages the ring cannot hold yet are near when it can
    if (seq_p < seq_s) {  // caught up by the stream: restart at its position
      fs_p = fs_s;
      p_p = p_s;
      seq_p = seq_s;
    }
    if (P.l2_window && fs_p < fs_c && (uint64_t)(seq_p - seq_s) * PG < P.l2_window) {
      const uint32_t f = fs_p % kFifo;
      const mk_instr &in = S.fifo[f];
      const uint32_t np = in.op == MK_OP_END ? 0u : S.meta[f].npages;
      if (p_p < np) {
        const void *gsrc;
        uint32_t bytes;
        page_src(P, S, in, p_p, np, gsrc, bytes);
        bulk_prefetch_l2(gsrc, bytes);
        ++p_p;
        ++seq_p;
        progress = true;
      }
      if (p_p >= np && in.op != MK_OP_END) {
        ++fs_p;
        p_p = 0;
      }
    }
    // ---- stream cursor
    if (fs_s < fs_c) {
      const uint32_t f = fs_s % kFifo;
      const mk_instr &in = S.fifo[f];
      if (in.op == MK_OP_END) break;  // everything before END is streamed
      const uint32_t np = S.meta[f].npages;
      if (p_s < np) {
        const uint32_t slot = seq_s % E, kk = seq_s / E;
        if (kk == 0 || mbar_test(&S.empty[slot], (kk - 1) & 1u)) {
          const void *gsrc;
          uint32_t bytes;
          page_src(P, S, in, p_s, np, gsrc, bytes);
          mbar_arrive_expect_tx(&S.full[slot], bytes);
          bulk_g2s(S.ring + (size_t)slot * PG, gsrc, bytes, &S.full[slot], pol);
          ++seq_s;
          ++p_s;
          progress = true;
        }
      }
      if (p_s == np) {
        if ((P.flags & MK_FLAG_TRACE) && np) S.meta[f].t_issued = gtimer();
        ++fs_s;
        p_s = 0;
        progress = true;
      }
    }
    if (progress) {
      t_idle = 0;
      n_idle = 0;
    } else {
      if (!t_idle) t_idle = cycles() | 1u;
      // idle: yield the sub-partition's issue slots to the compute warps on it
      __nanosleep(P.loader_idle_ns);
      if (should_stop(P, S, t_idle, n_idle, kWhereLoader | fs_s)) {
        ok = false;
        break;
      }
    }
  }
  if (!ok) drain_copies(P, S, seq_s);
}


DEVI void preload_gain_b1(const KParams &P, const mk_instr &in, uint32_t s, int lane,
                          XCache &X) {
  const OpGeom &G = P.geom[in.op];
  const uint16_t *gain = gain_of(P, in.op, in.layer);
  if (!gain) return;
#pragma unroll
  for (int j = 0; j < kMaxChunks; ++j)
    if (j < (int)G.nch) load_gain8(gain, s * G.SW + j * 256 + lane * 8, X.v[j]);
}


// Normalised inputs (QKV, gate/up, LM head) and the O-projection's input:
// all compute warps stage the K activations of the sequence into shared memory in one round trip, each
// adding its squares to a per-warp partial, then meet at a barrier.  The
// staging buffer is single: the next normalised phase depends (through the
// counters) on every instruction of this one, including this block's, so no
// warp still reads it when the next staging starts.
DEVI bool stages_input(const KParams &P, const mk_instr &in) {
  return in.op == MK_OP_OPROJ || gain_of(P, in.op, in.layer) != nullptr;
}

DEVI bool stage_input(const KParams &P, const Smem &S, const mk_instr &in, int cw, int lane,
                      uint32_t &xbar_uses) {
  const uint32_t K = P.geom[in.op].K;
  const int emb = in.op == MK_OP_QKV && (in.flags & 1);
  const float *src = in.op == MK_OP_OPROJ ? P.attn : P.x;
  float ss = 0.f;
  // every load of a thread is issued before the first is used, so the
  // staging costs one round trip to L2 (KS loads of 4 values per thread
  // cover K up to KS * 14 * 32 * 4 = 5376; a longer K takes more batches)
  constexpr int KS = 3;
  constexpr uint32_t kStride = kComputeWarps * 32 * 4;
  for (uint32_t i0 = (uint32_t)(cw * 32 + lane) * 4; i0 < K; i0 += KS * kStride) {
    float4 v[KS];
#pragma unroll
    for (int t = 0; t < KS; ++t) {
      const uint32_t i = i0 + t * kStride;
      v[t] = make_float4(0.f, 0.f, 0.f, 0.f);
      if (i < K) {
        if (emb) {
          const uint2 w =
              __ldg(reinterpret_cast<const uint2 *>(P.embed + (size_t)S.tok[0] * P.H + i));
          v[t] = make_float4(bf_lo(w.x), bf_hi(w.x), bf_lo(w.y), bf_hi(w.y));
        } else {
          v[t] = __ldcg(reinterpret_cast<const float4 *>(src + i));
        }
      }
    }
#pragma unroll
    for (int t = 0; t < KS; ++t) {
      const uint32_t i = i0 + t * kStride;
      if (i < K) *reinterpret_cast<float4 *>(S.xs + i) = v[t];
      ss = fmaf(v[t].x, v[t].x, fmaf(v[t].y, v[t].y, fmaf(v[t].z, v[t].z, fmaf(v[t].w, v[t].w, ss))));
    }
  }
  ss = warp_sum(ss);
  if (lane == 0) S.xs[K + cw] = ss;
  return compute_sync(P, S, S.xbar, xbar_uses, lane);
}

// After the dependency: the warp's input slice into registers.  X holds the
// gains (preloaded) for normalised inputs, which take x from shared memory.
DEVI void finish_input_b1(const KParams &P, const Smem &S, const mk_instr &in, uint32_t s,
                          int lane, XCache &X) {
  const OpGeom &G = P.geom[in.op];
  if (gain_of(P, in.op, in.layer) != nullptr) {
    float ss = 0.f;
    for (int w = 0; w < kComputeWarps; ++w) ss += S.xs[G.K + w];
    const float r = rsqrtf(ss / (float)G.K + P.eps);
#pragma unroll
    for (int j = 0; j < kMaxChunks; ++j)
      if (j < (int)G.nch) {
        const float *xp = S.xs + s * G.SW + j * 256 + lane * 8;
        const float4 a = *reinterpret_cast<const float4 *>(xp);
        const float4 c = *reinterpret_cast<const float4 *>(xp + 4);
        const float x8[8] = {a.x, a.y, a.z, a.w, c.x, c.y, c.z, c.w};
#pragma unroll
        for (int t = 0; t < 8; ++t) X.v[j][t] = x8[t] * r * X.v[j][t];
      }
    return;
  }
  if (in.op == MK_OP_OPROJ) {  // staged, no norm
#pragma unroll
    for (int j = 0; j < kMaxChunks; ++j)
      if (j < (int)G.nch) {
        const float *xp = S.xs + s * G.SW + j * 256 + lane * 8;
        const float4 a = *reinterpret_cast<const float4 *>(xp);
        const float4 c = *reinterpret_cast<const float4 *>(xp + 4);
        X.v[j][0] = a.x; X.v[j][1] = a.y; X.v[j][2] = a.z; X.v[j][3] = a.w;
        X.v[j][4] = c.x; X.v[j][5] = c.y; X.v[j][6] = c.z; X.v[j][7] = c.w;
      }
    return;
  }
#pragma unroll
  for (int j = 0; j < kMaxChunks; ++j)
    if (j < (int)G.nch) load8(P, S, in.op, 0, 0, s * G.SW + j * 256 + lane * 8, X.v[j]);
}

DEVI float dot_item_b1(const uint8_t *item, const XCache &X, int nch, int lane) {
  float a0 = 0.f, a1 = 0.f, a2 = 0.f, a3 = 0.f;
#pragma unroll
  for (int j = 0; j < kMaxChunks; ++j)
    if (j < nch) {
      const uint4 w = *reinterpret_cast<const uint4 *>(item + j * 512 + lane * 16);
      a0 = fmaf(bf_lo(w.x), X.v[j][0], a0);
      a1 = fmaf(bf_hi(w.x), X.v[j][1], a1);
      a2 = fmaf(bf_lo(w.y), X.v[j][2], a2);
      a3 = fmaf(bf_hi(w.y), X.v[j][3], a3);
      a0 = fmaf(bf_lo(w.z), X.v[j][4], a0);
      a1 = fmaf(bf_hi(w.z), X.v[j][5], a1);
      a2 = fmaf(bf_lo(w.w), X.v[j][6], a2);
      a3 = fmaf(bf_hi(w.w), X.v[j][7], a3);
    }
  return (a0 + a1) + (a2 + a3);
}

// FP8 weights: an item is SW E4M3 codes (one byte each); lane l's eight codes
// of chunk j are the same columns as in the bf16 item (j 256 + 8 l + t).
DEVI float2 e4m3x2_to_float2(uint32_t two) {
  const __half2_raw h = __nv_cvt_fp8x2_to_halfraw2((__nv_fp8x2_storage_t)two, __NV_E4M3);
  return __half22float2(__half2(h));
}

DEVI float dot_item_q8(const uint8_t *item, const XCache &X, int nch, int lane) {
  float a0 = 0.f, a1 = 0.f, a2 = 0.f, a3 = 0.f;
#pragma unroll
  for (int j = 0; j < kMaxChunks; ++j)
    if (j < nch) {
      const uint2 w = *reinterpret_cast<const uint2 *>(item + j * 256 + lane * 8);
      const float2 f0 = e4m3x2_to_float2(w.x & 0xFFFFu), f1 = e4m3x2_to_float2(w.x >> 16);
      const float2 f2 = e4m3x2_to_float2(w.y & 0xFFFFu), f3 = e4m3x2_to_float2(w.y >> 16);
      a0 = fmaf(f0.x, X.v[j][0], a0);
      a1 = fmaf(f0.y, X.v[j][1], a1);
      a2 = fmaf(f1.x, X.v[j][2], a2);
      a3 = fmaf(f1.y, X.v[j][3], a3);
      a0 = fmaf(f2.x, X.v[j][4], a0);
      a1 = fmaf(f2.y, X.v[j][5], a1);
      a2 = fmaf(f3.x, X.v[j][6], a2);
      a3 = fmaf(f3.y, X.v[j][7], a3);
    }
  return (a0 + a1) + (a2 + a3);
}

template <bool Q8>
DEVI float dot_item(const uint8_t *item, const XCache &X, int nch, int lane) {
  if constexpr (Q8) return dot_item_q8(item, X, nch, lane);
  else return dot_item_b1(item, X, nch, lane);
}

// Batch > 1: per-sequence 1/rms at every change of input, shared through
// shared memory (double-buffered by the change count).
DEVI bool norm_factors(const KParams &P, const Smem &S, const mk_instr &in, int cw, int lane,
                       uint32_t &xbar_uses, float *normr) {
  const OpGeom &G = P.geom[in.op];
  const int emb = in.op == MK_OP_QKV && (in.flags & 1);
  const bool norm = gain_of(P, in.op, in.layer) != nullptr;
  for (int b = cw; b < P.B; b += kComputeWarps) {  // a warp per sequence
    float r = 1.f;
    if (norm) {
      // normalised inputs are x or an embedding row
      float ss = 0.f;
      if (emb) {
        const uint16_t *row = P.embed + (size_t)S.tok[b] * P.H;
        for (uint32_t c = lane * 8; c < G.K; c += 512) {
          const uint4 w0 = __ldg(reinterpret_cast<const uint4 *>(row + c));
          const uint4 w1 = c + 256 < G.K ? __ldg(reinterpret_cast<const uint4 *>(row + c + 256))
                                         : make_uint4(0u, 0u, 0u, 0u);
          const uint32_t w[8] = {w0.x, w0.y, w0.z, w0.w, w1.x, w1.y, w1.z, w1.w};
#pragma unroll
          for (int t = 0; t < 8; ++t) {
            const float lo = bf_lo(w[t]), hi = bf_hi(w[t]);
            ss = fmaf(lo, lo, ss);
            ss = fmaf(hi, hi, ss);
          }
        }
      } else {
        const float *row = P.x + (size_t)b * P.H;
        for (uint32_t c = lane * 8; c < G.K; c += 1024) {  // 32 values of a lane in flight
          float4 q[8];
#pragma unroll
          for (int t = 0; t < 4; ++t) {
            const bool in_k = c + 256 * t < G.K;
            const float4 z = make_float4(0.f, 0.f, 0.f, 0.f);
            q[2 * t] = in_k ? __ldcg(reinterpret_cast<const float4 *>(row + c + 256 * t)) : z;
            q[2 * t + 1] = in_k ? __ldcg(reinterpret_cast<const float4 *>(row + c + 256 * t + 4)) : z;
          }
#pragma unroll
          for (int t = 0; t < 8; ++t) {
            ss = fmaf(q[t].x, q[t].x, ss);
            ss = fmaf(q[t].y, q[t].y, ss);
            ss = fmaf(q[t].z, q[t].z, ss);
            ss = fmaf(q[t].w, q[t].w, ss);
          }
        }
      }
      ss = warp_sum(ss);
      r = rsqrtf(ss / (float)G.K + P.eps);
    }
    if (lane == 0) normr[b] = r;
  }
  __syncwarp();
  if (lane == 0) mbar_arrive(S.xbar);
  const bool ok = warp_wait(P, S, S.xbar, xbar_uses & 1u, kWhereCompute);
  ++xbar_uses;
  return ok;
}

// Batch-1 GEMV of one instruction; X holds the normalised input slice when
// xkey matches the instruction's input.
template <bool Q8>
DEVI bool gemv_b1(const KParams &P, const Smem &S, const mk_instr &in, const SlotMeta &meta,
                  float *res, int cw, int lane, XCache &X, bool reload) {
  const OpGeom &G = P.geom[in.op];
  const uint32_t wrows = in.op == MK_OP_GATEUP ? 2 * in.nrows : in.nrows;
  const uint32_t items = wrows * G.NS;
  const uint32_t A = G.NS * (kComputeWarps / G.NS);
  const bool active = (uint32_t)cw < A;
  const uint32_t s = cw % G.NS;
  if (reload && active) finish_input_b1(P, S, in, s, lane, X);
  // trace stamps (compute warp 0): input in registers, first and last page present
  const bool stamp = cw == 0 && lane == 0 && (P.flags & MK_FLAG_TRACE);
  SlotMeta &mw = const_cast<SlotMeta &>(meta);  // meta is this entry's slot in shared memory
  if (stamp) mw.t_input = gtimer();
  const uint32_t E = P.ring_pages;
  uint32_t item = cw;
  for (uint32_t p = 0; p < meta.npages; ++p) {
    const uint32_t seq = meta.seq0 + p, slot = seq % E;
    if (!warp_wait(P, S, &S.full[slot], (seq / E) & 1u, kWhereCompute | meta.idx)) return false;
    if (stamp && p == 0) mw.t_page0 = gtimer();
    if (stamp && p + 1 == meta.npages) mw.t_pagel = gtimer();
    const uint8_t *page = S.ring + (size_t)slot * P.page_bytes;
    const uint32_t it_end = min(items, (p + 1) * G.ipp);
    // two items at a time where the page holds both: independent loads and
    // reductions overlap
    for (; active && item + A < it_end; item += 2 * A) {
      const uint8_t *ip = page + (item - p * G.ipp) * G.item_bytes;
      float a = dot_item<Q8>(ip, X, G.nch, lane);
      float c = dot_item<Q8>(ip + A * G.item_bytes, X, G.nch, lane);
#pragma unroll
      for (int o = 16; o; o >>= 1) {
        a += __shfl_xor_sync(0xFFFFFFFFu, a, o);
        c += __shfl_xor_sync(0xFFFFFFFFu, c, o);
      }
      if (lane == 0) {
        res[item] = a;
        res[item + A] = c;
      }
    }
    for (; active && item < it_end; item += A) {
      const uint8_t *ip = page + (item - p * G.ipp) * G.item_bytes;
      const float acc = warp_sum(dot_item<Q8>(ip, X, G.nch, lane));
      if (lane == 0) res[item] = acc;
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&S.empty[slot]);
  }
  return true;
}


// ---------------------------------------------- batch > 1: tensor cores ----
// The epilogue of a split projection block, run by the compute threads of the
// block's last slice: out(r, b) = the sum over slices, in slice order, of the
// slices' partial sums; then RoPE and the KV append (q/k/v rows), the
// residual (O, down), SiLU(gate) * up, or the logits.
__device__ __noinline__ bool tc_epilogue(const KParams &P, const Smem &S, const mk_instr &in,
                                         int tid, int lane, uint32_t &xbar_uses) {
  const OpGeom &G = P.geom[in.op];
  const int B = P.B, MR = (int)G.MR, NSL = (int)in.nchunk, d = P.d;
  const int rb = (int)in.row0 / (in.op == MK_OP_GATEUP ? MR / 2 : MR);
  const float *gp = P.gpart + (size_t)rb * NSL * MR * B;
  constexpr int T = kComputeWarps * 32;
  // 1. every (row, sequence) sum of the slices, in slice order, into shared
  //    memory (the attention scratch, idle during a projection): a thread's
  //    three outputs and four slices of each in flight at once, so the gather
  //    costs about one round trip to L2
  float *sums = S.opart;  // [MR][B]
  const int nsum = MR * B;
  for (int o0 = tid; o0 < nsum; o0 += 3 * T) {
    float v[3] = {0.f, 0.f, 0.f};
    for (int s0 = 0; s0 < NSL; s0 += 4) {
      float w[3][4];
#pragma unroll
      for (int k = 0; k < 3; ++k)
#pragma unroll
        for (int t = 0; t < 4; ++t)
          w[k][t] = (o0 + k * T < nsum && s0 + t < NSL)
                        ? __ldcg(gp + (size_t)(s0 + t) * MR * B + o0 + k * T) : 0.f;
#pragma unroll
      for (int k = 0; k < 3; ++k)
#pragma unroll
        for (int t = 0; t < 4; ++t) v[k] += w[k][t];
    }
#pragma unroll
    for (int k = 0; k < 3; ++k)
      if (o0 + k * T < nsum) sums[o0 + k * T] = v[k];
  }
  if (!compute_sync(P, S, S.xbar, xbar_uses, lane)) return false;
  auto val = [&](int r, int b) { return sums[r * B + b]; };
  switch (in.op) {
    case MK_OP_QKV: {
      const int GR = (P.qpg + 2) * d, half = d / 2, npairs = (int)in.nrows / 2;
      for (int u = tid; u < npairs * B; u += T) {
        const int pr = u % npairs, b = u / npairs;
        const int R = (int)in.row0 + 2 * pr, grp = R / GR, q = R % GR;
        const float x0 = val(2 * pr, b), x1 = val(2 * pr + 1, b);
        if (q < (P.qpg + 1) * d) {
          const int i = (q % d) / 2;
          const float cs = S.rope[b * d + i], sn = S.rope[b * d + half + i];
          const float o0 = x0 * cs - x1 * sn, o1 = x0 * sn + x1 * cs;
          if (q < P.qpg * d) {
            float *qd = P.q + ((size_t)b * P.nq + grp * P.qpg + q / d) * d;
            qd[i] = o0;
            qd[i + half] = o1;
          } else {
            uint16_t *kd = P.kc + kv_row(P, in.layer, b, grp, S.pos[b]);
            kd[i] = to_bf(o0);
            kd[i + half] = to_bf(o1);
          }
        } else {
          uint16_t *vd = P.vc + kv_row(P, in.layer, b, grp, S.pos[b]) + (q - (P.qpg + 1) * d);
          vd[0] = to_bf(x0);
          vd[1] = to_bf(x1);
        }
      }
      break;
    }
    case MK_OP_OPROJ:
    case MK_OP_DOWN: {
      const int n = (int)in.nrows * B;
      const bool emb = in.op == MK_OP_OPROJ && (in.flags & 1);
      for (int u0 = tid; u0 < n; u0 += 3 * T) {  // three residual loads in flight
        float resid[3];
#pragma unroll
        for (int k = 0; k < 3; ++k) {
          const int u = u0 + k * T;
          resid[k] = 0.f;
          if (u < n) {
            const int r = u % in.nrows, b = u / in.nrows, row = in.row0 + r;
            resid[k] = emb ? bf1(P.embed[(size_t)S.tok[b] * P.H + row])
                           : __ldcg(P.x + (size_t)b * P.H + row);
          }
        }
#pragma unroll
        for (int k = 0; k < 3; ++k) {
          const int u = u0 + k * T;
          if (u < n) {
            const int r = u % in.nrows, b = u / in.nrows, row = in.row0 + r;
            P.x[(size_t)b * P.H + row] = resid[k] + val(r, b);
          }
        }
      }
      break;
    }
    case MK_OP_GATEUP:  // rows interleave gate j (2j) and up j (2j + 1)
      for (int u = tid; u < (int)in.nrows * B; u += T) {
        const int j = u % in.nrows, b = u / in.nrows;
        const float gt = val(2 * j, b), up = val(2 * j + 1, b);
        P.h[(size_t)b * P.F + in.row0 + j] = gt / (1.f + __expf(-gt)) * up;
      }
      break;
    default:  // LM head
      for (int u = tid; u < (int)in.nrows * B; u += T) {
        const int r = u % in.nrows, b = u / in.nrows;
        P.logits[(size_t)b * P.V + in.row0 + r] = val(r, b);
      }
      break;
  }
  return true;
}

// One batch > 1 projection tile: MR weight rows x the input columns of
// slice `chunk` of `nchunk` (whole pages of kc columns), on the tensor cores.
//  1. Compute warps 1.. stage the MMA's B operand page by page into a ring
//     of kTcBufs shared-memory slots, kTcBufs - 2 pages ahead of the MMAs:
//     the page's columns of the B (normalised) input rows as bf16 values in
//     rows 0..B-1 and as bf16 remainders x - bf16(x) in rows B..2B-1, so
//     value plus remainder keep about 16 significant bits of the fp32 input.
//     A slot is refilled once the commit of the MMAs that read it lands.
//  2. Compute warp 0 lane 0 issues the MMAs (A = the ring page, K-major,
//     fp32 accumulator in tensor memory) page by page as weight page and B
//     slot land; a commit releases each page once its MMAs are done (the
//     other warps' arrivals make up the rest of the page's release count).
//  3. The four warps whose ids cover the four lane quarters of tensor memory
//     read the MR x N accumulator and add value and remainder columns: an
//     unsplit LM-head or gate/up tile writes its logits or SiLU(gate) * up
//     from there; other tiles write these partial sums to global memory.
//  4. An unsplit tile that wrote partial sums runs tc_epilogue itself; a
//     split tile arrives on its block's counter (acq_rel) and the last slice
//     runs tc_epilogue over the slices' sums.  Either releases the phase
//     counter.
__device__ __noinline__ bool gemv_tc(const KParams &P, const Smem &S, const mk_instr &in,
                                     const SlotMeta &meta, int cw, int lane, uint32_t epoch,
                                     uint32_t &xkey, uint32_t &xbar_uses, uint32_t &key_changes,
                                     uint32_t &tc_uses, uint32_t &bseq) {
  const OpGeom &G = P.geom[in.op];
  const int B = P.B, NB = P.tc_nb, MR = (int)G.MR, kc = (int)G.kc;
  const int tid = cw * 32 + lane;
  const int emb = in.op == MK_OP_QKV && (in.flags & 1);
  const uint16_t *gain = gain_of(P, in.op, in.layer);
  uint8_t *bop = reinterpret_cast<uint8_t *>(S.xs);
  const uint32_t slot_bytes = (uint32_t)kc * (uint32_t)NB * 2u;
  const int c0 = in.nchunk > 1 ? (int)(in.chunk * G.kp / in.nchunk) * kc : 0;
  const uint32_t where = kWhereCompute | meta.idx, np = meta.npages, b0 = bseq;
  // producer geometry (step 1 below); a producer's first page of activations
  // is fetched before the norm factors, so the two round trips overlap
  const int units = B * (kc / 8), pt = tid - 32;
  const int NG = ((kComputeWarps - 1) * 32) / units;  // >= 1 (checked by the planner)
  const int grp = pt >= 0 ? pt / units : NG;
  const bool has = grp < NG;
  const int ub = has ? (pt % units) / (kc / 8) : 0, uk = has ? (pt % (kc / 8)) * 8 : 0;
  float v[8];
  auto fetch = [&](uint32_t q) {
    if (has && q < np) load8(P, S, in.op, emb, ub, c0 + (int)q * kc + uk, v);
  };
  if (cw != 0) fetch((uint32_t)grp);
  const uint32_t key = input_key(in);
  if (key != xkey) {
    ++key_changes;
    if (!norm_factors(P, S, in, cw, lane, xbar_uses, S.normr + (key_changes & 1u) * kMaxBatch))
      return false;
    xkey = key;
  }
  const float *normr = S.normr + (key_changes & 1u) * kMaxBatch;
  // 1. B operand of page q (rows >= 2B stay zero from the kernel's start),
  //    written by compute warps 1.. (warp 0 issues the MMAs).  The producer
  //    threads form NG groups of one (sequence, 8 columns) unit each; group
  //    g owns pages g, g + NG, ... and fetches its next page's activations
  //    right after storing one, so each fetch has NG pages' time to land.
  //    Every producer warp arrives on every slot (after the wait for the
  //    slot's previous MMAs), so a slot's count never depends on ownership.
  auto store = [&](uint32_t q) -> bool {
    const uint32_t n = b0 + q, bs = n % kTcBufs;
    if (n >= (uint32_t)kTcBufs &&
        !warp_wait(P, S, &S.bempty[bs], (n / kTcBufs - 1u) & 1u, where))
      return false;
    if (has && (int)(q % (uint32_t)NG) == grp) {
      uint8_t *dst = bop + bs * slot_bytes;
      const float r = normr[ub];
      float g8[8];
      if (gain) load_gain8(gain, c0 + (int)q * kc + uk, g8);
      uint32_t hi[4], lo[4];
#pragma unroll
      for (int u = 0; u < 8; u += 2) {
        const float x0 = v[u] * r * (gain ? g8[u] : 1.f);
        const float x1 = v[u + 1] * r * (gain ? g8[u + 1] : 1.f);
        const uint16_t h0 = to_bf(x0), h1 = to_bf(x1);
        const uint16_t l0 = to_bf(x0 - bf1(h0)), l1 = to_bf(x1 - bf1(h1));
        hi[u / 2] = (uint32_t)h0 | ((uint32_t)h1 << 16);
        lo[u / 2] = (uint32_t)l0 | ((uint32_t)l1 << 16);
      }
      const int kb = (uk / 16) * (NB * 32) + ((uk / 8) % 2) * 128;
      *reinterpret_cast<uint4 *>(dst + kb + (ub / 8) * 256 + (ub % 8) * 16) =
          make_uint4(hi[0], hi[1], hi[2], hi[3]);
      *reinterpret_cast<uint4 *>(dst + kb + ((B + ub) / 8) * 256 + ((B + ub) % 8) * 16) =
          make_uint4(lo[0], lo[1], lo[2], lo[3]);
      fetch(q + (uint32_t)NG);
    }
    fence_proxy_async();  // generic-proxy writes become visible to the tensor cores
    __syncwarp();
    if (lane == 0) mbar_arrive(&S.bfull[bs]);
    return true;
  };
  if (cw != 0) {
    // 2a. producers: every page's slot, in order (at most kTcBufs ahead of
    //     the MMAs through the slots' release; the first fetch went out above)
    for (uint32_t q = 0; q < np; ++q)
      if (!store(q)) return false;
  } else {
    // 2b. MMAs: page p once its weights and its B slot are in; the commit
    //     releases both (the page's only release in tensor-core plans)
    const uint32_t E = P.ring_pages, taddr = (uint32_t)S.misc[3];
    const uint32_t idesc = tc_idesc((uint32_t)MR, (uint32_t)NB);
    const bool stamp = lane == 0 && (P.flags & MK_FLAG_TRACE);
    SlotMeta &mw = const_cast<SlotMeta &>(meta);  // this entry's slot in shared memory
    if (stamp) mw.t_input = gtimer();
    for (uint32_t p = 0; p < np; ++p) {
      const uint32_t seq = meta.seq0 + p, slot = seq % E;
      const uint32_t n = b0 + p, bs = n % kTcBufs;
      if (!warp_wait(P, S, &S.full[slot], (seq / E) & 1u, where)) return false;
      if (stamp && p == 0) mw.t_page0 = gtimer();
      if (!warp_wait(P, S, &S.bfull[bs], (n / kTcBufs) & 1u, where)) return false;
      if (stamp && p + 1 == np) mw.t_pagel = gtimer();
      if (lane == 0) {
        tc_fence_after();
        const uint32_t abase = saddr(S.ring + (size_t)slot * P.page_bytes);
        const uint32_t bbase = saddr(bop + bs * slot_bytes);
        for (uint32_t t = 0; t < (uint32_t)kc / 16; ++t)
          tc_mma(taddr, tc_desc(abase + t * (uint32_t)MR * 32, 128, 256),
                 tc_desc(bbase + t * (uint32_t)NB * 32, 128, 256), idesc, (p | t) != 0);
        tc_commit(&S.empty[slot]);
        tc_commit(&S.bempty[bs]);
      }
      __syncwarp();
    }
  }
  bseq = b0 + np;
  const uint32_t taddr = (uint32_t)S.misc[3];
  // an unsplit LM-head or gate/up tile writes its outputs straight from the
  // accumulator; other tiles go through the partial-sum buffer
  const bool unsplit = in.sig2_ctr == MK_NO_COUNTER;
  const bool direct = unsplit && (in.op == MK_OP_LMHEAD || in.op == MK_OP_GATEUP);
  if (cw == 0 && lane == 0) tc_commit(S.tbar);
  // 3. accumulator -> partial sums (warp w of the block reads lanes 32 (w % 4) ..)
  if (cw >= 2 && cw < 6) {
    const int qd = (cw + 2) % 4;
    if (!warp_wait(P, S, S.tbar, tc_uses & 1u, kWhereCompute | meta.idx)) return false;
    if (32 * qd < MR) {
      tc_fence_after();
      const uint32_t ta = taddr + ((uint32_t)(32 * qd) << 16);
      const int r = 32 * qd + lane;
      const int rb = (int)in.row0 / (in.op == MK_OP_GATEUP ? MR / 2 : MR);
      float *gdst = P.gpart + (((size_t)rb * in.nchunk + in.chunk) * MR + r) * B;
      // one output (row r, sequence b) = value column b + remainder column B + b
      auto emit = [&](int b, float x) {
        if (direct && in.op == MK_OP_LMHEAD) {
          if (r < (int)in.nrows) P.logits[(size_t)b * P.V + in.row0 + r] = x;
        } else if (direct) {  // gate/up: lane 2j holds gate j, lane 2j + 1 up j
          const int jg = r / 2;
          const float up = __shfl_xor_sync(0xFFFFFFFFu, x, 1);
          if (!(lane & 1) && jg < (int)in.nrows)
            P.h[(size_t)b * P.F + in.row0 + jg] = x / (1.f + __expf(-x)) * up;
        } else {
          gdst[b] = x;
        }
      };
      if (B <= 16) {  // values and remainders within the first 32 columns
        float v[32];
        float(&v0)[16] = *reinterpret_cast<float(*)[16]>(v);
        float(&v1)[16] = *reinterpret_cast<float(*)[16]>(v + 16);
        tc_ld16(ta, v0);
        if (NB > 16) tc_ld16(ta + 16, v1);
#pragma unroll
        for (int b = 0; b < 16; ++b)
          if (b < B) emit(b, v[b] + v[B + b]);
      } else {  // B a multiple of 16: sixteen sequences' values and remainders at a time
        for (int b0 = 0; b0 < B; b0 += 16) {
          float va[16], vr[16];
          tc_ld16(ta + (uint32_t)b0, va);
          tc_ld16(ta + (uint32_t)(B + b0), vr);
#pragma unroll
          for (int b = 0; b < 16; ++b) emit(b0 + b, va[b] + vr[b]);
        }
      }
    }
  }
  ++tc_uses;
  tc_fence_before();
  if (!compute_sync(P, S, S.xbar, xbar_uses, lane)) return false;
  if (unsplit) {  // the tile owns its rows: finish them and signal the phase
    if (!direct) {
      if (!tc_epilogue(P, S, in, tid, lane, xbar_uses)) return false;
      if (!compute_sync(P, S, S.xbar, xbar_uses, lane)) return false;
    }
    if (cw == 0 && lane == 0) red_release(P.ctr + (size_t)in.sig_ctr * kCtrStride, 1u);
    return true;
  }
  // 4. arrival; the block's last slice sums the slices and finishes the rows
  if (cw == 0 && lane == 0) {
    const uint32_t old = atom_add_acq_rel(P.ctr + (size_t)in.sig_ctr * kCtrStride, 1u);
    S.misc[2] = old == epoch * in.nchunk + in.nchunk - 1u ? 1 : 0;
  }
  if (!compute_sync(P, S, S.xbar, xbar_uses, lane)) return false;
  if (S.misc[2]) {
    if (!tc_epilogue(P, S, in, tid, lane, xbar_uses)) return false;
    if (!compute_sync(P, S, S.xbar, xbar_uses, lane)) return false;
    if (cw == 0 && lane == 0) red_release(P.ctr + (size_t)in.sig2_ctr * kCtrStride, 1u);
  }
  return true;
}

// Step 6 of an attention chunk, shared by both chunk layouts: the chunk's
// partial {m, l, o} is in global memory (written before the block barrier
// this starts with); take the arrival and, for the group's last chunk, merge.
template <int D, int QPG>
__device__ __forceinline__ bool attn_arrive_merge(const KParams &P, const Smem &S,
                                                  const mk_instr &in, int cw, int lane,
                                                  uint32_t &att_uses, uint32_t epoch, int b,
                                                  int g, int pos) {
  // arrival: the chunk that completes its (sequence, group) merges all of
  //    the group's chunk partials by log-sum-exp, in chunk order, with every
  //    compute thread (one output each), and
  //    releases the group counter.  The acq_rel arrival publishes this chunk's
  //    partial (ordered before it by the barrier) and, for the last arriver,
  //    acquires every other chunk's.
  //    Only the nch chunks that reach p_b arrive: the last of them also adds
  //    the nchunk - nch empty chunks' share, so the counter still advances by
  //    nchunk per step.
  const int nch = min((int)in.nchunk, (pos + P.attn_chunk) / P.attn_chunk);
  if (!compute_sync(P, S, S.attbar, att_uses, lane)) return false;
  if (cw == 0 && lane == 0) {
    uint32_t *ctr = P.ctr + (size_t)in.sig_ctr * kCtrStride;
    const uint32_t old = atom_add_acq_rel(ctr, 1u);
    const bool last = old == epoch * in.nchunk + (uint32_t)nch - 1u;
    if (last && (uint32_t)nch < in.nchunk) red_add(ctr, in.nchunk - (uint32_t)nch);
    S.misc[2] = last ? 1 : 0;
  }
  if (!compute_sync(P, S, S.attbar, att_uses, lane)) return false;
  if (S.misc[2]) {
    const int PS = 2 * QPG + QPG * D;
    const float *pb = P.part + ((size_t)b * P.nkv + g) * in.nchunk * PS;
    // up to MB chunks' partials in flight at once (one round trip to L2 for
    // a group of up to MB chunks); per batch, the batch's maximum first, then
    // one rescale of the running sums
    constexpr int MB = 16;
    for (int o = cw * 32 + lane; o < QPG * D; o += kComputeWarps * 32) {
      const int h = o / D;
      float M = -INFINITY, den = 0.f, num = 0.f;
      for (int c0 = 0; c0 < nch; c0 += MB) {
        float mc[MB], lc[MB], oc[MB];
#pragma unroll
        for (int u = 0; u < MB; ++u) {
          mc[u] = -INFINITY;
          lc[u] = oc[u] = 0.f;
          if (c0 + u < nch) {
            const float *pc = pb + (size_t)(c0 + u) * PS;
            mc[u] = __ldcg(pc + h);
            lc[u] = __ldcg(pc + QPG + h);
            oc[u] = __ldcg(pc + 2 * QPG + o);
          }
        }
        float Mb = M;
#pragma unroll
        for (int u = 0; u < MB; ++u) Mb = fmaxf(Mb, mc[u]);
        if (Mb == -INFINITY) continue;
        const float a = __expf(M - Mb);
        den *= a;
        num *= a;
#pragma unroll
        for (int u = 0; u < MB; ++u) {
          if (mc[u] == -INFINITY) continue;
          const float w = __expf(mc[u] - Mb);
          den = fmaf(w, lc[u], den);
          num = fmaf(w, oc[u], num);
        }
        M = Mb;
      }
      P.attn[(size_t)b * P.nq * D + (size_t)g * QPG * D + o] = num / den;
    }
    if (!compute_sync(P, S, S.attbar, att_uses, lane)) return false;
    if (cw == 0 && lane == 0) red_release(P.ctr + (size_t)in.sig2_ctr * kCtrStride, 1u);
  }
  return true;
}

// One split-KV attention chunk for the QPG query heads of group g of
// sequence b over its positions [p0, p1): scores q.k/sqrt(d), the chunk's
// maximum m, denominator l = sum exp(s - m) and unnormalised output
// o = sum exp(s - m) v, written to the partials buffer as {m[QPG], l[QPG],
// o[QPG][D]} (the paper's split-KV decode attention; chunks are merged by
// log-sum-exp once all of a group's chunks are in).
//
// Keys and values of the positions below p_b arrive as one ring page each;
// the key and value of p_b itself (written this step) are read from global
// memory.  Warp cw serves head cw % QPG over a contiguous share of the
// chunk: it keeps its scores in its own shared-memory row, so the warps meet
// only once, to merge the per-warp partials of each head.
template <int D, int QPG>
__device__ __noinline__ bool attn_chunk(const KParams &P, const Smem &S, const mk_instr &in,
                                        const SlotMeta &meta, int cw, int lane,
                                        uint32_t &att_uses, uint32_t epoch) {
  constexpr int LPP = D / 8;      // lanes per key row (16 bytes each)
  constexpr int RPS = 32 / LPP;   // key rows per warp step
  constexpr int DPL = D / 32;     // value dims per lane
  const int b = in.b, g = in.g, pos = S.pos[b];
  int p0, p1;
  attn_range(P, pos, in.chunk, p0, p1);
  const int n_tot = p1 - p0;
  const int n_old = max(0, min(p1, pos) - p0);  // rows that come from the ring
  const uint32_t E = P.ring_pages;
  const int h = cw % QPG, r = cw / QPG;
  const int nqs = (kComputeWarps - 1 - h) / QPG + 1;  // warps serving head h
  const int len = (n_tot + nqs - 1) / nqs;
  const int j0 = min(r * len, n_tot), j1 = min(j0 + len, n_tot);
  const int part = lane % LPP;
  const bool stamp = cw == 0 && lane == 0 && (P.flags & MK_FLAG_TRACE);
  SlotMeta &mw = const_cast<SlotMeta &>(meta);  // this entry's slot in shared memory
  // A chunk past p_b has nothing to do: it neither computes nor arrives (the
  // group's last real chunk adds the empty chunks' share of the arrivals).
  if (n_tot <= 0) return true;

  // query slice of head h (8 dims per lane), pre-scaled by 1/sqrt(d); the
  // current position's key slice and value dims if this warp covers p_b
  float q8[8], kn8[8], vn[DPL];
  {
    const float *qh = P.q + ((size_t)b * P.nq + (size_t)g * QPG + h) * D + part * 8;
    const float4 x0 = __ldcg(reinterpret_cast<const float4 *>(qh));
    const float4 x1 = __ldcg(reinterpret_cast<const float4 *>(qh + 4));
    const float sc = P.attn_scale;
    q8[0] = x0.x * sc; q8[1] = x0.y * sc; q8[2] = x0.z * sc; q8[3] = x0.w * sc;
    q8[4] = x1.x * sc; q8[5] = x1.y * sc; q8[6] = x1.z * sc; q8[7] = x1.w * sc;
#pragma unroll
    for (int u = 0; u < 8; ++u) kn8[u] = 0.f;
#pragma unroll
    for (int k = 0; k < DPL; ++k) vn[k] = 0.f;
    if (n_old >= j0 && n_old < j1) {
      const size_t at = kv_row(P, in.layer, b, g, pos);
      const uint4 w = __ldcg(reinterpret_cast<const uint4 *>(P.kc + at + part * 8));
      kn8[0] = bf_lo(w.x); kn8[1] = bf_hi(w.x); kn8[2] = bf_lo(w.y); kn8[3] = bf_hi(w.y);
      kn8[4] = bf_lo(w.z); kn8[5] = bf_hi(w.z); kn8[6] = bf_lo(w.w); kn8[7] = bf_hi(w.w);
#pragma unroll
      for (int k = 0; k < DPL; ++k) vn[k] = bf1(__ldcg(P.vc + at + lane * DPL + k));
    }
  }
  if (stamp) mw.t_input = gtimer();
  const bool paged = n_old > 0;  // one key page and one value page
  const uint8_t *__restrict__ kpage = S.ring + (size_t)(meta.seq0 % E) * P.page_bytes;
  const uint8_t *__restrict__ vpage = S.ring + (size_t)((meta.seq0 + 1) % E) * P.page_bytes;
  if (paged && !warp_wait(P, S, &S.full[meta.seq0 % E], (meta.seq0 / E) & 1u, kWhereCompute | meta.idx))
    return false;

  // 1. scores of rows j0..j1 into this warp's row of S.sc.  A block of LPP
  //    steps covers 32 rows; each lane keeps its LPP partial dot products and
  //    one transposing butterfly over the LPP lanes of a row group leaves
  //    lane `part` with the full score of step `part` (LPP - 1 shuffles for
  //    LPP rows instead of log2(LPP) per row).
  float *__restrict__ sw = S.sc + (size_t)cw * P.att_lmax;
  for (int jb = j0; jb < j1; jb += LPP * RPS) {
    float v[LPP];
#pragma unroll
    for (int t = 0; t < LPP; ++t) {
      const int j = jb + t * RPS + lane / LPP;
      float k8[8];
      if (j < n_old) {
        const uint4 w = *reinterpret_cast<const uint4 *>(kpage + (size_t)j * D * 2 + part * 16);
        k8[0] = bf_lo(w.x); k8[1] = bf_hi(w.x); k8[2] = bf_lo(w.y); k8[3] = bf_hi(w.y);
        k8[4] = bf_lo(w.z); k8[5] = bf_hi(w.z); k8[6] = bf_lo(w.w); k8[7] = bf_hi(w.w);
      } else {
        const bool cur = j < j1;  // the row of p_b itself
#pragma unroll
        for (int u = 0; u < 8; ++u) k8[u] = cur ? kn8[u] : 0.f;
      }
      float a0 = 0.f, a1 = 0.f;
#pragma unroll
      for (int u = 0; u < 8; u += 2) {
        a0 = fmaf(q8[u], k8[u], a0);
        a1 = fmaf(q8[u + 1], k8[u + 1], a1);
      }
      v[t] = a0 + a1;
    }
#pragma unroll
    for (int hw = LPP / 2; hw >= 1; hw /= 2) {
      const bool upper = (part & hw) != 0;
#pragma unroll
      for (int i = 0; i < hw; ++i) {
        const float send = upper ? v[i] : v[i + hw];
        const float keep = upper ? v[i + hw] : v[i];
        v[i] = keep + __shfl_xor_sync(0xFFFFFFFFu, send, hw);
      }
    }
    const int jr = jb + part * RPS + lane / LPP;
    if (jr < j1) sw[jr - j0] = v[0];
  }
  __syncwarp();
  if (stamp) mw.t_page0 = gtimer();

  // 2. this warp's maximum, probabilities and denominator
  const int cnt = j1 - j0;
  float mx = -INFINITY;
  for (int i = lane; i < cnt; i += 32) mx = fmaxf(mx, sw[i]);
  const float m = warp_max(mx);
  float lsum = 0.f;
  for (int i = lane; i < cnt; i += 32) {
    const float pj = __expf(sw[i] - m);
    sw[i] = pj;
    lsum += pj;
  }
  const float l = warp_sum(lsum);
  __syncwarp();

  // 3. o = sum_j p_j v_j over this warp's rows; lanes own DPL dims each
  if (paged && !warp_wait(P, S, &S.full[(meta.seq0 + 1) % E], ((meta.seq0 + 1) / E) & 1u,
                          kWhereCompute | meta.idx))
    return false;
  if (stamp) mw.t_pagel = gtimer();
  float o[8][DPL];
#pragma unroll
  for (int u = 0; u < 8; ++u)
#pragma unroll
    for (int k = 0; k < DPL; ++k) o[u][k] = 0.f;
  const int jo = min(j1, n_old);  // rows of this warp that come from the value page
  const uint8_t *__restrict__ vrow = vpage + lane * DPL * 2;
  int j = j0;
  // eight positions per iteration: two 16-byte loads of probabilities (the
  // warp's score row is 16-byte aligned and j - j0 steps by 8) and eight
  // independent accumulators
  for (; j + 8 <= jo; j += 8) {
    const float4 pa = *reinterpret_cast<const float4 *>(sw + (j - j0));
    const float4 pb = *reinterpret_cast<const float4 *>(sw + (j - j0) + 4);
    const float pj[8] = {pa.x, pa.y, pa.z, pa.w, pb.x, pb.y, pb.z, pb.w};
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const uint8_t *row = vrow + (size_t)(j + u) * D * 2;
      if constexpr (DPL == 2) {
        const uint32_t w = *reinterpret_cast<const uint32_t *>(row);
        o[u][0] = fmaf(pj[u], bf_lo(w), o[u][0]);
        o[u][1] = fmaf(pj[u], bf_hi(w), o[u][1]);
      } else {
        const uint2 w = *reinterpret_cast<const uint2 *>(row);
        o[u][0] = fmaf(pj[u], bf_lo(w.x), o[u][0]);
        o[u][1] = fmaf(pj[u], bf_hi(w.x), o[u][1]);
        o[u][DPL > 2 ? 2 : 0] = fmaf(pj[u], bf_lo(w.y), o[u][DPL > 2 ? 2 : 0]);
        o[u][DPL > 2 ? 3 : 1] = fmaf(pj[u], bf_hi(w.y), o[u][DPL > 2 ? 3 : 1]);
      }
    }
  }
  for (; j < j1; ++j) {
    const float pj = sw[j - j0];
    if (j < n_old) {
      const uint8_t *row = vrow + (size_t)j * D * 2;
#pragma unroll
      for (int k = 0; k < DPL; k += 2) {
        const uint32_t w = *reinterpret_cast<const uint32_t *>(row + k * 2);
        o[0][k] = fmaf(pj, bf_lo(w), o[0][k]);
        o[0][k + 1] = fmaf(pj, bf_hi(w), o[0][k + 1]);
      }
    } else {
#pragma unroll
      for (int k = 0; k < DPL; ++k) o[0][k] = fmaf(pj, vn[k], o[0][k]);
    }
  }
  // every warp is done with the chunk's pages
  __syncwarp();
  if (paged && !P.tc && lane == 0) {
    mbar_arrive(&S.empty[meta.seq0 % E]);
    mbar_arrive(&S.empty[(meta.seq0 + 1) % E]);
  }

  // 4. per-warp partials (double-buffered by instruction parity: a warp can
  //    be at most one instruction ahead of the warps merging the last one)
  const uint32_t par = att_uses & 1u;
  float *op = S.opart + (size_t)par * kComputeWarps * D;
  float *mlp = S.ml + par * kComputeWarps * 2;
#pragma unroll
  for (int k = 0; k < DPL; ++k)
    op[cw * D + lane * DPL + k] =
        ((o[0][k] + o[1][k]) + (o[2][k] + o[3][k])) + ((o[4][k] + o[5][k]) + (o[6][k] + o[7][k]));
  if (lane == 0) {
    mlp[cw * 2] = m;
    mlp[cw * 2 + 1] = l;
  }
  if (!compute_sync(P, S, S.attbar, att_uses, lane)) return false;
  if (paged && P.tc && cw == 0 && lane == 0) {  // every warp is past the pages
    mbar_arrive(&S.empty[meta.seq0 % E]);
    mbar_arrive(&S.empty[(meta.seq0 + 1) % E]);
  }

  // 5. warp hh < QPG merges the partials of head hh into the chunk partial
  if (cw < QPG) {
    float M = -INFINITY;
    for (int w = cw; w < kComputeWarps; w += QPG) M = fmaxf(M, mlp[w * 2]);
    float L = 0.f, acc[DPL];
#pragma unroll
    for (int k = 0; k < DPL; ++k) acc[k] = 0.f;
    if (M != -INFINITY) {
      for (int w = cw; w < kComputeWarps; w += QPG) {
        const float mw_ = mlp[w * 2];
        if (mw_ == -INFINITY) continue;
        const float a = __expf(mw_ - M);
        L = fmaf(a, mlp[w * 2 + 1], L);
#pragma unroll
        for (int k = 0; k < DPL; ++k) acc[k] = fmaf(a, op[w * D + lane * DPL + k], acc[k]);
      }
    }
    const int PS = 2 * QPG + QPG * D;
    float *dst = P.part + (((size_t)b * P.nkv + g) * P.nchunk + in.chunk) * PS;
#pragma unroll
    for (int k = 0; k < DPL; ++k) dst[2 * QPG + cw * D + lane * DPL + k] = acc[k];
    if (lane == 0) {
      dst[cw] = M;
      dst[QPG + cw] = L;
    }
  }

  // 6. arrival, and the group merge by its last chunk
  return attn_arrive_merge<D, QPG>(P, S, in, cw, lane, att_uses, epoch, b, g, pos);
}

// The same chunk for tensor-core plans with d = 64 and at most four query
// heads per group: the chunk's positions are split over all compute warps,
// and each warp scores its rows for every head of the group, so every key
// and value row is read from shared memory once (by one warp) instead of
// once per head, and every warp has the same number of rows.  Scores are
// kept as [row][head]; the per-warp partials {o[head][d]}, {m, l}[head] are
// single-buffered: the per-head merge reads them before the barrier that
// precedes the arrival, which every warp passes before it can reach the next
// chunk.
// MP: the chunk may span several key (and value) pages (chunks longer than
// a page); otherwise every row is in the chunk's one key and one value page.
template <int QPG, bool MP>
__device__ __noinline__ bool attn_chunk_grp(const KParams &P, const Smem &S, const mk_instr &in,
                                            const SlotMeta &meta, int cw, int lane,
                                            uint32_t &att_uses, uint32_t epoch) {
  constexpr int D = 64;
  constexpr int LPP = D / 8;      // lanes per key row (16 bytes each)
  constexpr int RPS = 32 / LPP;   // key rows per warp step
  constexpr int DPL = D / 32;     // value dims per lane
  const int b = in.b, g = in.g, pos = S.pos[b];
  int p0, p1;
  attn_range(P, pos, in.chunk, p0, p1);
  const int n_tot = p1 - p0;
  const int n_old = max(0, min(p1, pos) - p0);  // rows that come from the ring
  const uint32_t E = P.ring_pages;
  const int len = (n_tot + kComputeWarps - 1) / kComputeWarps;
  const int j0 = min(cw * len, n_tot), j1 = min(j0 + len, n_tot);
  const int part = lane % LPP;
  const bool stamp = cw == 0 && lane == 0 && (P.flags & MK_FLAG_TRACE);
  SlotMeta &mw = const_cast<SlotMeta &>(meta);  // this entry's slot in shared memory
  if (n_tot <= 0) return true;
  float *op = S.opart;                                  // [warp][head][D]
  float *mlp = op + kComputeWarps * QPG * D;            // [warp][head][m, l]
  float *sw = mlp + kComputeWarps * QPG * 2 + (size_t)cw * P.att_lmax;  // [row][head]

  // queries of every head (8 dims per lane), pre-scaled; the current
  // position's key slice and value dims if this warp covers p_b
  float q8[QPG][8], kn8[8], vn[DPL];
  {
    const float sc = P.attn_scale;
#pragma unroll
    for (int h = 0; h < QPG; ++h) {
      const float *qh = P.q + ((size_t)b * P.nq + (size_t)g * QPG + h) * D + part * 8;
      const float4 x0 = __ldcg(reinterpret_cast<const float4 *>(qh));
      const float4 x1 = __ldcg(reinterpret_cast<const float4 *>(qh + 4));
      q8[h][0] = x0.x * sc; q8[h][1] = x0.y * sc; q8[h][2] = x0.z * sc; q8[h][3] = x0.w * sc;
      q8[h][4] = x1.x * sc; q8[h][5] = x1.y * sc; q8[h][6] = x1.z * sc; q8[h][7] = x1.w * sc;
    }
#pragma unroll
    for (int u = 0; u < 8; ++u) kn8[u] = 0.f;
#pragma unroll
    for (int k = 0; k < DPL; ++k) vn[k] = 0.f;
    if (n_old >= j0 && n_old < j1) {
      const size_t at = kv_row(P, in.layer, b, g, pos);
      const uint4 w = __ldcg(reinterpret_cast<const uint4 *>(P.kc + at + part * 8));
      kn8[0] = bf_lo(w.x); kn8[1] = bf_hi(w.x); kn8[2] = bf_lo(w.y); kn8[3] = bf_hi(w.y);
      kn8[4] = bf_lo(w.z); kn8[5] = bf_hi(w.z); kn8[6] = bf_lo(w.w); kn8[7] = bf_hi(w.w);
#pragma unroll
      for (int k = 0; k < DPL; ++k) vn[k] = bf1(__ldcg(P.vc + at + lane * DPL + k));
    }
  }
  if (stamp) mw.t_input = gtimer();
  // keys of the cached rows arrive as npk ring pages of rpp rows each (a power
  // of two), then their values as npk more; a warp's rows span at most two
  // pages, whose addresses it works out once
  const int rs = __ffs((int)P.page_bytes / (D * 2)) - 1, rpp = 1 << rs;
  const int npk = (n_old + rpp - 1) >> rs;
  const bool paged = n_old > 0;
  const int pg0 = j0 >> rs;
  const uint8_t *base[2][2];
#pragma unroll
  for (int side = 0; side < 2; ++side)
#pragma unroll
    for (int k = 0; k < (MP ? 2 : 1); ++k) {
      const uint32_t seq = meta.seq0 + (uint32_t)(MP ? side * npk + pg0 + k : side);
      base[side][k] = S.ring + (size_t)(seq % E) * P.page_bytes;
    }
  auto row_ptr = [&](int side, int j) {  // side 0 keys, 1 values; j0 <= j < n_old
    if (!MP) return base[side][0] + (size_t)j * D * 2;  // pg0 = 0, one page per side
    return base[side][(j >> rs) - pg0] + (size_t)(j & (rpp - 1)) * D * 2;
  };
  auto wait_rows = [&](int side) -> bool {  // the pages holding rows j0 .. j1 - 1
    if (!MP) {
      if (!paged) return true;
      const uint32_t seq = meta.seq0 + (uint32_t)side;
      return warp_wait(P, S, &S.full[seq % E], (seq / E) & 1u, kWhereCompute | meta.idx);
    }
    const int jl = min(j1, n_old);
    if (j0 >= jl) return true;
    for (int pg = j0 / rpp; pg <= (jl - 1) / rpp; ++pg) {
      const uint32_t seq = meta.seq0 + (uint32_t)(side * npk + pg);
      if (!warp_wait(P, S, &S.full[seq % E], (seq / E) & 1u, kWhereCompute | meta.idx))
        return false;
    }
    return true;
  };
  if (!wait_rows(0)) return false;

  // 1. scores of rows j0..j1 for every head: a block of LPP steps covers 32
  //    rows; per head one transposing butterfly over the LPP lanes of a row
  //    group leaves lane `part` with the full score of step `part`.  Steps t
  //    and t + LPP/2 are scored together and take the butterfly's first level
  //    at once, so only half the steps' partial sums are live per head.
  auto score8 = [&](int j, float (&out)[QPG]) {
    float k8[8];
    if (j < n_old) {
      const uint4 w = *reinterpret_cast<const uint4 *>(row_ptr(0, j) + part * 16);
      k8[0] = bf_lo(w.x); k8[1] = bf_hi(w.x); k8[2] = bf_lo(w.y); k8[3] = bf_hi(w.y);
      k8[4] = bf_lo(w.z); k8[5] = bf_hi(w.z); k8[6] = bf_lo(w.w); k8[7] = bf_hi(w.w);
    } else {
      const bool cur = j < j1;  // the row of p_b itself
#pragma unroll
      for (int u = 0; u < 8; ++u) k8[u] = cur ? kn8[u] : 0.f;
    }
#pragma unroll
    for (int h = 0; h < QPG; ++h) {
      float a0 = 0.f, a1 = 0.f;
#pragma unroll
      for (int u = 0; u < 8; u += 2) {
        a0 = fmaf(q8[h][u], k8[u], a0);
        a1 = fmaf(q8[h][u + 1], k8[u + 1], a1);
      }
      out[h] = a0 + a1;
    }
  };
  constexpr int HALF = LPP / 2;
  for (int jb = j0; jb < j1; jb += LPP * RPS) {
    float v[QPG][HALF];
    const bool up4 = (part & HALF) != 0;
#pragma unroll
    for (int t = 0; t < HALF; ++t) {
      float va[QPG], vb[QPG];
      score8(jb + t * RPS + lane / LPP, va);
      score8(jb + (t + HALF) * RPS + lane / LPP, vb);
#pragma unroll
      for (int h = 0; h < QPG; ++h) {
        const float send = up4 ? va[h] : vb[h];
        const float keep = up4 ? vb[h] : va[h];
        v[h][t] = keep + __shfl_xor_sync(0xFFFFFFFFu, send, HALF);
      }
    }
#pragma unroll
    for (int hw = HALF / 2; hw >= 1; hw /= 2) {
      const bool upper = (part & hw) != 0;
#pragma unroll
      for (int h = 0; h < QPG; ++h)
#pragma unroll
        for (int i = 0; i < hw; ++i) {
          const float send = upper ? v[h][i] : v[h][i + hw];
          const float keep = upper ? v[h][i + hw] : v[h][i];
          v[h][i] = keep + __shfl_xor_sync(0xFFFFFFFFu, send, hw);
        }
    }
    const int jr = jb + part * RPS + lane / LPP;
    if (jr < j1)
#pragma unroll
      for (int h = 0; h < QPG; ++h) sw[(jr - j0) * QPG + h] = v[h][0];
  }
  __syncwarp();
  if (stamp) mw.t_page0 = gtimer();

  // 2. per head: this warp's maximum, probabilities and denominator
  const int cnt = j1 - j0;  // at most 32 rows per warp (chunks of <= 448 positions)
  float m[QPG], l[QPG];
#pragma unroll
  for (int h = 0; h < QPG; ++h) {
    const float s = lane < cnt ? sw[lane * QPG + h] : -INFINITY;
    m[h] = warp_max(s);
    const float pj = lane < cnt ? __expf(s - m[h]) : 0.f;
    if (lane < cnt) sw[lane * QPG + h] = pj;
    l[h] = warp_sum(pj);
  }
  __syncwarp();

  // 3. o[h] = sum_j p_j[h] v_j over this warp's rows; lanes own DPL dims,
  //    even and odd rows in separate accumulators
  if (!wait_rows(1)) return false;
  if (stamp) mw.t_pagel = gtimer();
  float o[2][QPG][DPL];
#pragma unroll
  for (int e = 0; e < 2; ++e)
#pragma unroll
    for (int h = 0; h < QPG; ++h)
#pragma unroll
      for (int k = 0; k < DPL; ++k) o[e][h][k] = 0.f;
  for (int j = j0; j < j1; j += 2) {
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      const int jj = j + e;
      if (jj < j1) {
        float vv[DPL];
        if (jj < n_old) {
          const uint32_t w = *reinterpret_cast<const uint32_t *>(row_ptr(1, jj) + lane * DPL * 2);
          vv[0] = bf_lo(w);
          vv[1] = bf_hi(w);
        } else {
#pragma unroll
          for (int k = 0; k < DPL; ++k) vv[k] = vn[k];
        }
        float pj[QPG];
        if constexpr (QPG == 4) {
          const float4 p4 = *reinterpret_cast<const float4 *>(sw + (jj - j0) * QPG);
          pj[0] = p4.x; pj[1] = p4.y; pj[2] = p4.z; pj[3] = p4.w;
        } else {
#pragma unroll
          for (int h = 0; h < QPG; ++h) pj[h] = sw[(jj - j0) * QPG + h];
        }
#pragma unroll
        for (int h = 0; h < QPG; ++h)
#pragma unroll
          for (int k = 0; k < DPL; ++k) o[e][h][k] = fmaf(pj[h], vv[k], o[e][h][k]);
      }
    }
  }

  // 4. per-warp partials, then one block barrier
#pragma unroll
  for (int h = 0; h < QPG; ++h) {
#pragma unroll
    for (int k = 0; k < DPL; ++k)
      op[((size_t)cw * QPG + h) * D + lane * DPL + k] = o[0][h][k] + o[1][h][k];
    if (lane == 0) {
      mlp[(cw * QPG + h) * 2] = cnt > 0 ? m[h] : -INFINITY;
      mlp[(cw * QPG + h) * 2 + 1] = l[h];
    }
  }
  if (!compute_sync(P, S, S.attbar, att_uses, lane)) return false;
  if (paged && cw == 0 && lane == 0) {  // every warp is past the pages
    if (MP) {
      for (int pg = 0; pg < 2 * npk; ++pg) mbar_arrive(&S.empty[(meta.seq0 + (uint32_t)pg) % E]);
    } else {
      mbar_arrive(&S.empty[meta.seq0 % E]);
      mbar_arrive(&S.empty[(meta.seq0 + 1) % E]);
    }
  }

  // 5. warp hh < QPG merges the partials of head hh into the chunk partial
  if (cw < QPG) {
    float M = -INFINITY;
    for (int w = 0; w < kComputeWarps; ++w) M = fmaxf(M, mlp[(w * QPG + cw) * 2]);
    float L = 0.f, acc[DPL];
#pragma unroll
    for (int k = 0; k < DPL; ++k) acc[k] = 0.f;
    if (M != -INFINITY) {
      for (int w = 0; w < kComputeWarps; ++w) {
        const float mw_ = mlp[(w * QPG + cw) * 2];
        if (mw_ == -INFINITY) continue;
        const float a = __expf(mw_ - M);
        L = fmaf(a, mlp[(w * QPG + cw) * 2 + 1], L);
#pragma unroll
        for (int k = 0; k < DPL; ++k)
          acc[k] = fmaf(a, op[((size_t)w * QPG + cw) * D + lane * DPL + k], acc[k]);
      }
    }
    const int PS = 2 * QPG + QPG * D;
    float *dst = P.part + (((size_t)b * P.nkv + g) * P.nchunk + in.chunk) * PS;
#pragma unroll
    for (int k = 0; k < DPL; ++k) dst[2 * QPG + cw * D + lane * DPL + k] = acc[k];
    if (lane == 0) {
      dst[cw] = M;
      dst[QPG + cw] = L;
    }
  }

  // 6. the chunk partial is in global memory once every warp is past this
  //    barrier (which also frees the per-warp partials for the next chunk);
  //    the storer takes the arrival and, for the group's last chunk, merges
  (void)epoch;
  return compute_sync(P, S, S.attbar, att_uses, lane);
}

template <bool TC>
DEVI bool attn_dispatch(const KParams &P, const Smem &S, const mk_instr &in,
                        const SlotMeta &meta, int cw, int lane, uint32_t &att_uses,
                        uint32_t epoch) {
  if constexpr (TC) {
    if (P.att_grp) {
      if (P.attn_chunk > (int)P.page_bytes / 128) {
        switch (P.qpg) {
          case 1: return attn_chunk_grp<1, true>(P, S, in, meta, cw, lane, att_uses, epoch);
          case 2: return attn_chunk_grp<2, true>(P, S, in, meta, cw, lane, att_uses, epoch);
          default: return attn_chunk_grp<4, true>(P, S, in, meta, cw, lane, att_uses, epoch);
        }
      }
      switch (P.qpg) {
        case 1: return attn_chunk_grp<1, false>(P, S, in, meta, cw, lane, att_uses, epoch);
        case 2: return attn_chunk_grp<2, false>(P, S, in, meta, cw, lane, att_uses, epoch);
        default: return attn_chunk_grp<4, false>(P, S, in, meta, cw, lane, att_uses, epoch);
      }
    }
  }
  if (P.d == 64) {
    switch (P.qpg) {
      case 1: return attn_chunk<64, 1>(P, S, in, meta, cw, lane, att_uses, epoch);
      case 2: return attn_chunk<64, 2>(P, S, in, meta, cw, lane, att_uses, epoch);
      case 4: return attn_chunk<64, 4>(P, S, in, meta, cw, lane, att_uses, epoch);
      default: return attn_chunk<64, 8>(P, S, in, meta, cw, lane, att_uses, epoch);
    }
  }
  switch (P.qpg) {
    case 1: return attn_chunk<128, 1>(P, S, in, meta, cw, lane, att_uses, epoch);
    case 2: return attn_chunk<128, 2>(P, S, in, meta, cw, lane, att_uses, epoch);
    case 4: return attn_chunk<128, 4>(P, S, in, meta, cw, lane, att_uses, epoch);
    default: return attn_chunk<128, 8>(P, S, in, meta, cw, lane, att_uses, epoch);
  }
}


// Batch-1 run of consecutive GEMV instructions sharing the register input
// cache; returns at the first attention or end entry (not consumed).
template <bool Q8>
DEVI bool run_gemv_b1(const KParams &P, const Smem &S, uint32_t &fs, uint32_t epoch, int cw,
                      int lane, uint32_t &xbar_uses) {
  XCache X;
  uint32_t xkey = 0xFFFFFFFFu;
  while (true) {
    const uint32_t f = fs % kFifo;
    const mk_instr &in = S.fifo[f];
    const SlotMeta &meta = S.meta[f];
    const uint32_t key = input_key(in);
    const bool reload = key != xkey;
    const uint32_t ns = P.geom[in.op].NS;
    if (reload && (uint32_t)cw < ns * (kComputeWarps / ns))
      preload_gain_b1(P, in, cw % ns, lane, X);
    xkey = key;
    if (!ready_entry(P, S, fs, in, meta, epoch, cw, lane)) return false;
    if (reload && stages_input(P, in) && !stage_input(P, S, in, cw, lane, xbar_uses))
      return false;
    if (!gemv_b1<Q8>(P, S, in, meta, S.res + (size_t)f * P.res_floats, cw, lane, X, reload))
      return false;
    finish_entry(P, S, fs, cw, lane);
    ++fs;
    if (!next_entry(P, S, fs)) return false;
    const uint8_t op = S.fifo[fs % kFifo].op;
    if (op == MK_OP_ATTN || op == MK_OP_END) return true;
  }
}

// The compute warps' loop.  Batch-1 plans run every projection as a CUDA-core
// GEMV; batch > 1 plans run them on the tensor cores.  The two are separate
// instantiations (and kernels), so neither's registers are shaped by the
// other's calls.
template <bool TC, bool Q8>
DEVI void compute(const KParams &P, const Smem &S, uint32_t epoch, int cw, int lane) {
  uint32_t att_uses = 0, xbar_uses = 0, key_changes = 0, xkey = 0xFFFFFFFFu, tc_uses = 0;
  uint32_t tc_bseq = 0, fs = 0;
  if (!next_entry(P, S, fs)) return;
  while (true) {
    const uint32_t f = fs % kFifo;
    const mk_instr &in = S.fifo[f];
    const SlotMeta &meta = S.meta[f];
    if (in.op == MK_OP_END) {
      finish_entry(P, S, fs, cw, lane);
      return;
    }
    if (!TC && in.op != MK_OP_ATTN) {
      if (!run_gemv_b1<Q8>(P, S, fs, epoch, cw, lane, xbar_uses)) return;
      continue;
    }
    if (!ready_entry(P, S, fs, in, meta, epoch, cw, lane)) return;
    bool ok;
    if (in.op == MK_OP_ATTN) {
      ok = attn_dispatch<TC>(P, S, in, meta, cw, lane, att_uses, epoch);
      xkey = 0xFFFFFFFFu;
    } else if (TC) {
      ok = gemv_tc(P, S, in, meta, cw, lane, epoch, xkey, xbar_uses, key_changes, tc_uses,
                   tc_bseq);
    } else {
      ok = false;
    }
    if (!ok) return;
    finish_entry(P, S, fs, cw, lane);
    ++fs;
    if (!next_entry(P, S, fs)) return;
  }
}


// Tensor-core plans with grouped attention: the storer warp takes a chunk's
// arrival off the compute warps (which go on to their next instruction once
// the chunk partial is written), and merges the group when its chunk is the
// last to arrive.  The compute warps' partial writes are ordered before the
// arrival through the slot's done barrier (the compute warps' release at CTA
// scope, this warp's acquire) and the arrival's own gpu-scope release.  The
// merge by one warp: lane c holds the maxima and denominators of chunk
// c0 + c for every head; each lane owns OPL consecutive outputs of one head
// and accumulates them over the chunks, CB chunks' loads in flight.
template <int QPG>
__device__ __noinline__ void storer_attn_grp(const KParams &P, const Smem &S, const mk_instr &in,
                                             int lane, uint32_t epoch) {
  constexpr int D = 64, PS = 2 * QPG + QPG * D, OPL = QPG * D / 32, CB = 4;
  const int b = in.b, g = in.g, pos = S.pos[b];
  int p0, p1;
  attn_range(P, pos, in.chunk, p0, p1);
  if (p1 - p0 <= 0) return;  // past p_b: no arrival (the last real chunk adds it)
  const int nch = min((int)in.nchunk, (pos + P.attn_chunk) / P.attn_chunk);
  int last = 0;
  if (lane == 0) {
    uint32_t *ctr = P.ctr + (size_t)in.sig_ctr * kCtrStride;
    const uint32_t old = atom_add_acq_rel(ctr, 1u);
    last = old == epoch * in.nchunk + (uint32_t)nch - 1u ? 1 : 0;
    if (last && (uint32_t)nch < in.nchunk) red_add(ctr, in.nchunk - (uint32_t)nch);
  }
  if (!__shfl_sync(0xFFFFFFFFu, last, 0)) return;
  const float *pb = P.part + ((size_t)b * P.nkv + g) * in.nchunk * PS;
  const int o0 = lane * OPL, hl = o0 / D;
  float M[QPG], den[QPG], num[OPL];
#pragma unroll
  for (int h = 0; h < QPG; ++h) {
    M[h] = -INFINITY;
    den[h] = 0.f;
  }
#pragma unroll
  for (int k = 0; k < OPL; ++k) num[k] = 0.f;
  for (int c0 = 0; c0 < nch; c0 += 32) {
    const int c = c0 + lane;
    const bool valid = c < nch;
    float w[QPG], a[QPG];
#pragma unroll
    for (int h = 0; h < QPG; ++h) {
      const float mh = valid ? __ldcg(pb + (size_t)c * PS + h) : -INFINITY;
      const float lh = valid ? __ldcg(pb + (size_t)c * PS + QPG + h) : 0.f;
      const float Mn = fmaxf(M[h], warp_max(mh));
      a[h] = M[h] == -INFINITY ? 0.f : __expf(M[h] - Mn);
      w[h] = mh == -INFINITY ? 0.f : __expf(mh - Mn);
      den[h] = den[h] * a[h] + warp_sum(w[h] * lh);
      M[h] = Mn;
    }
    float ah = a[0];
#pragma unroll
    for (int h = 1; h < QPG; ++h) ah = hl == h ? a[h] : ah;
#pragma unroll
    for (int k = 0; k < OPL; ++k) num[k] *= ah;
    const int nb = min(32, nch - c0);
    for (int cb = 0; cb < nb; cb += CB) {
      float oc[CB][OPL];
#pragma unroll
      for (int u = 0; u < CB; ++u)
        if (cb + u < nb) {
          const float *src = pb + (size_t)(c0 + cb + u) * PS + 2 * QPG + o0;
#pragma unroll
          for (int k = 0; k < OPL; k += 4) {
            const float4 v = __ldcg(reinterpret_cast<const float4 *>(src + k));
            oc[u][k] = v.x; oc[u][k + 1] = v.y; oc[u][k + 2] = v.z; oc[u][k + 3] = v.w;
          }
        }
#pragma unroll
      for (int u = 0; u < CB; ++u)
        if (cb + u < nb) {
          float wu = 0.f;
#pragma unroll
          for (int h = 0; h < QPG; ++h) {
            const float wh = __shfl_sync(0xFFFFFFFFu, w[h], cb + u);
            wu = hl == h ? wh : wu;
          }
#pragma unroll
          for (int k = 0; k < OPL; ++k) num[k] = fmaf(wu, oc[u][k], num[k]);
        }
    }
  }
  float dh = den[0];
#pragma unroll
  for (int h = 1; h < QPG; ++h) dh = hl == h ? den[h] : dh;
  float *dst = P.attn + (size_t)b * P.nq * D + (size_t)g * QPG * D + o0;
#pragma unroll
  for (int k = 0; k < OPL; ++k) dst[k] = num[k] / dh;
  __syncwarp();
  if (lane == 0) red_release(P.ctr + (size_t)in.sig2_ctr * kCtrStride, 1u);
}

// FP8 plans: the row scales of a batch-1 tile follow its pages in the arena
DEVI void prefetch_scales(const KParams &P, const Smem &S, const mk_instr &in, int lane) {
  if (in.op == MK_OP_ATTN) return;
  const uint32_t w = in.op == MK_OP_GATEUP ? 2 * in.nrows : in.nrows;
  const float *sc =
      reinterpret_cast<const float *>(P.arena + in.wofs + (uint64_t)in.npages * P.page_bytes);
  for (uint32_t r = lane; r < w; r += 32) S.wsc[r] = __ldg(sc + r);
}

template <bool TC, bool Q8>
DEVI void storer(const KParams &P, const Smem &S, uint32_t epoch, int lane) {
  for (uint32_t fs = 0;; ++fs) {
    const uint32_t f = fs % kFifo, k = fs / kFifo;
    if (!warp_wait(P, S, &S.ifull[f], k & 1u, kWhereStorer)) break;
    const mk_instr &in = S.fifo[f];
    const SlotMeta &meta = S.meta[f];
    if (in.op == MK_OP_END) break;
    if (!warp_wait(P, S, &S.rdy[f], k & 1u, kWhereStorer)) break;
    if (!P.tc) prefetch_residual(P, S, in, lane);
    if (Q8) prefetch_scales(P, S, in, lane);
    if (!warp_wait(P, S, &S.done[f], k & 1u, kWhereStorer)) break;
    if (lane == 0 && (P.flags & MK_FLAG_TRACE)) S.meta[f].t_sstart = gtimer();
    __syncwarp();
    if (TC && P.att_grp && in.op == MK_OP_ATTN) {
      switch (P.qpg) {
        case 1: storer_attn_grp<1>(P, S, in, lane, epoch); break;
        case 2: storer_attn_grp<2>(P, S, in, lane, epoch); break;
        default: storer_attn_grp<4>(P, S, in, lane, epoch); break;
      }
      __syncwarp();
    }
    storer_epilogue<Q8>(P, S, in, meta, S.res + (size_t)f * P.res_floats, lane, epoch);
    __syncwarp();
    if (lane == 0) mbar_arrive(&S.iempty[f]);
  }
}

// --------------------------------------------------------------- kernel ----
template <bool TC, bool Q8>
DEVI void megakernel_body(const KParams &P) {
  extern __shared__ __align__(1024) uint8_t smem[];
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  // The table of shared-memory pointers lives in shared memory itself: a
  // per-thread copy would sit in local memory, which the small L1 left
  // beside a full shared-memory carve-out cannot hold for 512 threads.
  Smem *desc = reinterpret_cast<Smem *>(smem + P.off_misc + kMiscDescOffset);
  if (tid == 0) *desc = make_smem(P, smem);
  __syncthreads();
  const Smem &S = *desc;
  if (tid == 0) {
    for (uint32_t i = 0; i < P.ring_pages; ++i) {
      mbar_init(&S.full[i], 1);
      // tensor-core plans: a page's one release is the MMA commit (a
      // projection) or compute warp 0 after the block's barrier (attention)
      mbar_init(&S.empty[i], P.tc ? 1 : kComputeWarps);
    }
    for (int i = 0; i < kFifo; ++i) {
      mbar_init(&S.ifull[i], 1);
      mbar_init(&S.iempty[i], 1);
      mbar_init(&S.rdy[i], 1);
      mbar_init(&S.done[i], kComputeWarps);
    }
    mbar_init(S.attbar, kComputeWarps);
    mbar_init(S.xbar, kComputeWarps);
    mbar_init(S.tbar, 1);
    mbar_init(S.dbar, 1);
    for (int i = 0; i < kTcBufs; ++i) {
      mbar_init(&S.bfull[i], kComputeWarps - 1);
      mbar_init(&S.bempty[i], 1);
    }
    fence_mbar_init();
    S.misc[0] = 0;
    S.misc[1] = 0;
  }
  for (int i = tid; i < P.n_wait; i += kThreads) S.sat[i] = 0u;
  const uint32_t epoch = ld_relaxed(P.ctrl + kCtlEpoch);
  __syncthreads();
  if (tid < P.B) {
    const int t = P.tokens[tid], p = P.positions[tid];
    S.tok[tid] = t;
    S.pos[tid] = p;
    if (t < 0 || t >= P.V || p < 0 || p >= P.max_ctx) S.misc[1] = 1;
  }
  __syncthreads();
  if (TC && P.nchunk <= kMaxDealChunks) {
    // the attention re-deal's tables for this launch's positions (the same
    // for every layer): chunk c has work for sequence b when p_b >= c * chunk
    for (int c = tid; c < P.nchunk; c += kThreads) {
      uint64_t m = 0;
      for (int b = 0; b < P.B; ++b)
        if (S.pos[b] >= c * P.attn_chunk) m |= 1ull << b;
      S.dmask[c] = m;
    }
    __syncthreads();
    if (tid == 0) {
      uint32_t acc = 0;
      for (int c = 0; c < P.nchunk; ++c) {
        S.dpre[c] = acc;
        acc += (uint32_t)__popcll(S.dmask[c]);
      }
      S.dpre[P.nchunk] = acc;
    }
    __syncthreads();
  }
  const bool bad = S.misc[1] != 0;
  if (!bad) {
    const int half = P.d / 2;
    for (int i = tid; i < P.B * half; i += kThreads) {
      const int b = i / half, k = i % half;
      const size_t at = (size_t)S.pos[b] * half + k;
      S.rope[b * P.d + k] = P.rope_cos[at];
      S.rope[b * P.d + half + k] = P.rope_sin[at];
    }
  }
  __syncthreads();
  if (bad) {
    if (tid == 0 && blockIdx.x == 0) raise_error(P, MK_ERR_BOUNDS, 0, false);
    return;
  }
  if (TC) {
    // tensor memory for the projections' accumulator (tmem_cols fp32
    // columns, a power of two >= 32 covering the 2B value and remainder
    // columns), and a zeroed B-operand buffer (rows past 2B stay zero)
    if (warp == 2) {
      asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                       saddr((const void *)(S.misc + 3))), "r"(P.tmem_cols)
                   : "memory");
      asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    uint32_t bop_bytes = 0;
    for (int op = MK_OP_QKV; op <= MK_OP_LMHEAD; ++op)
      if (op != MK_OP_ATTN)
        bop_bytes = max(bop_bytes, kTcBufs * P.geom[op].kc * (uint32_t)P.tc_nb * 2u);
    for (uint32_t i = tid; i < bop_bytes / 16; i += kThreads)
      reinterpret_cast<uint4 *>(S.xs)[i] = make_uint4(0u, 0u, 0u, 0u);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
  }
  if (warp == 0) {
    if (lane == 0) {
      if (P.mode == kModeHybrid) loader<TC, true>(P, S, epoch);
      else loader<TC, false>(P, S, epoch);
    }
    __syncwarp();
  } else if (warp == 1) {
    storer<TC, Q8>(P, S, epoch, lane);
  } else {
    compute<TC, Q8>(P, S, epoch, warp - 2, lane);
  }
  __syncthreads();
  if (TC) {
    // every tensor-core operation (issued by compute warp 0 lane 0) is done
    // before the accumulator's tensor memory is freed
    if (warp == 2 && lane == 0) {
      tc_commit(S.dbar);
      const uint64_t t0 = cycles();
      while (!mbar_try_wait(S.dbar, 0u))
        if (cycles() - t0 > P.timeout_cycles) {
          raise_error(P, MK_ERR_TIMEOUT, kWhereDrain | 0xFFFFFFu, true);
          break;
        }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 2)
      asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"((uint32_t)S.misc[3]),
                   "r"(P.tmem_cols)
                   : "memory");
  }
  // a block only bails after a latched error; never let it end silently
  if (tid == 0 && S.misc[0] != 0) raise_error(P, MK_ERR_TIMEOUT, 0x0FFFFFFFu, true);
  if (tid == 0 && P.mode != kModeRange && S.misc[0] == 0) {
    fence_gpu();
    const uint32_t old = atomicAdd(P.ctrl + kCtlExit, 1u);
    if (old == epoch * P.n_blocks + P.n_blocks - 1u) atomicExch(P.ctrl + kCtlEpoch, epoch + 1u);
  }
}

// Batch-1 plans (CUDA-core GEMVs) and batch > 1 plans (tensor-core
// projections): the same persistent interpreter, compiled twice.
extern "C" __global__ void __launch_bounds__(kThreads, 1)
    mk_megakernel(const __grid_constant__ KParams P) {
  megakernel_body<false, false>(P);
}
extern "C" __global__ void __launch_bounds__(kThreads, 1)
    mk_megakernel_tc(const __grid_constant__ KParams P) {
  megakernel_body<true, false>(P);
}
// Batch-1 plans with FP8 weights (MK_FLAG_FP8_WEIGHTS)
extern "C" __global__ void __launch_bounds__(kThreads, 1)
    mk_megakernel_q8(const __grid_constant__ KParams P) {
  megakernel_body<false, true>(P);
}

// The multi-kernel path ends each step with this one-thread launch.
extern "C" __global__ void mk_epoch_advance(uint32_t *ctrl) { ctrl[kCtlEpoch] += 1u; }

// Re-tiling of one weight block: tile-row k of a block whose source row is
// Arena row k takes source row map[k] (k when map is NULL), split into NS
// items of item_bytes packed ipp per page; rowtab[k] = byte offset of its
// tile | its row within the tile (tiles are page-aligned, rows < 4096).
extern "C" __global__ void mk_retile(uint8_t *dst, const uint8_t *src, const int32_t *map,
                                     const uint64_t *rowtab, uint32_t nrows, uint32_t K,
                                     uint32_t NS, uint32_t item_bytes, uint32_t ipp,
                                     uint32_t page) {
  const uint64_t per_row = (uint64_t)K * 2 / 16;
  const uint64_t total = (uint64_t)nrows * per_row;
  for (uint64_t i = (uint64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total;
       i += (uint64_t)gridDim.x * blockDim.x) {
    const uint32_t k = (uint32_t)(i / per_row);
    const uint32_t cb = (uint32_t)(i % per_row) * 16;
    const uint32_t s = cb / item_bytes, ib = cb % item_bytes;
    const uint64_t rt = rowtab[k];
    const uint32_t r = (uint32_t)(rt & 4095u);
    const uint32_t item = r * NS + s;
    uint8_t *d = dst + (rt & ~(uint64_t)4095u) + (uint64_t)(item / ipp) * page +
                 (uint64_t)(item % ipp) * item_bytes + ib;
    const uint32_t srow = map ? (uint32_t)map[k] : k;
    *reinterpret_cast<uint4 *>(d) =
        *reinterpret_cast<const uint4 *>(src + (uint64_t)srow * K * 2 + cb);
  }
}

// Tensor-core blocks (batch > 1 plans): weight row k (source row map[k]) and
// 8 columns from c go to block rb = k / MR (row rr = k % MR), page c / kc of
// the block's kp pages along K, and inside the page to the core matrix
// (rr / 8, (cc / 8) % 2) of k-step cc / 16, cc = c % kc: the MMA reads a
// k-step as MR x 16 bf16 in 8-row x 16-byte core matrices, 128 bytes apart
// along K and 256 bytes apart along M.
extern "C" __global__ void mk_retile_tc(uint8_t *dst, const uint8_t *src, const int32_t *map,
                                        uint32_t nrows, uint32_t K, uint32_t MR, uint32_t kc,
                                        uint32_t kp, uint32_t page) {
  const uint64_t per_row = K / 8;
  const uint64_t total = (uint64_t)nrows * per_row;
  for (uint64_t i = (uint64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total;
       i += (uint64_t)gridDim.x * blockDim.x) {
    const uint32_t k = (uint32_t)(i / per_row);
    const uint32_t c = (uint32_t)(i % per_row) * 8;
    const uint32_t rb = k / MR, rr = k % MR, j = c / kc, cc = c % kc;
    uint8_t *d = dst + ((uint64_t)rb * kp + j) * page + (cc / 16) * (MR * 32) +
                 (rr / 8) * 256 + ((cc / 8) % 2) * 128 + (rr % 8) * 16;
    const uint32_t srow = map ? (uint32_t)map[k] : k;
    *reinterpret_cast<uint4 *>(d) =
        *reinterpret_cast<const uint4 *>(src + (uint64_t)srow * K * 2 + (uint64_t)c * 2);
  }
}

// FP8 plans, step 1 of re-tiling a weight block: arena row k's scale, the
// largest magnitude of source row map[k] over 448 (1 for a zero row), at
// byte scaletab[k] of the block.  One warp per row.
extern "C" __global__ void mk_row_scale(uint8_t *dst, const uint8_t *src, const int32_t *map,
                                        const uint64_t *scaletab, uint32_t nrows, uint32_t K) {
  const int lane = threadIdx.x & 31;
  const uint32_t warps = gridDim.x * (blockDim.x / 32);
  for (uint32_t k = blockIdx.x * (blockDim.x / 32) + threadIdx.x / 32; k < nrows; k += warps) {
    const uint32_t srow = map ? (uint32_t)map[k] : k;
    const uint16_t *row = reinterpret_cast<const uint16_t *>(src) + (uint64_t)srow * K;
    float amax = 0.f;
    for (uint32_t c = lane; c < K; c += 32) amax = fmaxf(amax, fabsf(bf1(row[c])));
    amax = warp_max(amax);
    if (lane == 0)
      *reinterpret_cast<float *>(dst + scaletab[k]) = amax > 0.f ? __fdiv_rn(amax, 448.0f) : 1.0f;
  }
}

// Step 2: the codes.  Eight columns per thread: code = E4M3 of w / scale
// (the division correctly rounded in float, the conversion to nearest even
// and saturating), written at the columns' place in their item (SW bytes
// per item, ipp items per page), as the bf16 re-tiling places 2 SW bytes.
extern "C" __global__ void mk_retile_q8(uint8_t *dst, const uint8_t *src, const int32_t *map,
                                        const uint64_t *rowtab, const uint64_t *scaletab,
                                        uint32_t nrows, uint32_t K, uint32_t NS,
                                        uint32_t item_bytes, uint32_t ipp, uint32_t page) {
  const uint64_t per_row = K / 8;
  const uint64_t total = (uint64_t)nrows * per_row;
  const uint32_t SW = K / NS;
  for (uint64_t i = (uint64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total;
       i += (uint64_t)gridDim.x * blockDim.x) {
    const uint32_t k = (uint32_t)(i / per_row);
    const uint32_t c = (uint32_t)(i % per_row) * 8;
    const uint64_t rt = rowtab[k];
    const uint32_t r = (uint32_t)(rt & 4095u);
    const uint32_t item = r * NS + c / SW;
    uint8_t *d = dst + (rt & ~(uint64_t)4095u) + (uint64_t)(item / ipp) * page +
                 (uint64_t)(item % ipp) * item_bytes + c % SW;
    const float sc = *reinterpret_cast<const float *>(dst + scaletab[k]);
    const uint32_t srow = map ? (uint32_t)map[k] : k;
    const uint4 w = *reinterpret_cast<const uint4 *>(src + ((uint64_t)srow * K + c) * 2);
    const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
    uint32_t out[2] = {0u, 0u};
#pragma unroll
    for (int t = 0; t < 8; ++t) {
      const uint32_t h = (ws[t / 2] >> (16 * (t % 2))) & 0xFFFFu;
      const float v = __fdiv_rn(__uint_as_float(h << 16), sc);
      const uint32_t q = (uint32_t)__nv_cvt_float_to_fp8(v, __NV_SATFINITE, __NV_E4M3);
      out[t / 4] |= q << (8 * (t % 4));
    }
    *reinterpret_cast<uint2 *>(d) = make_uint2(out[0], out[1]);
  }
}

// ---- host-side launch helpers (the kernels' host stubs live in this unit) ----
cudaError_t set_megakernel_smem(uint32_t bytes) {
  cudaError_t e = cudaFuncSetAttribute(mk_megakernel_tc,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(mk_megakernel_q8, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           (int)bytes);
  if (e != cudaSuccess) return e;
  return cudaFuncSetAttribute(mk_megakernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              (int)bytes);
}

cudaError_t launch_megakernel(const KParams &P, uint32_t grid, bool cooperative,
                              cudaStream_t stream) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = P.smem_total;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = cooperative ? 1 : 0;
  return P.tc    ? cudaLaunchKernelEx(&cfg, mk_megakernel_tc, P)
         : P.fp8 ? cudaLaunchKernelEx(&cfg, mk_megakernel_q8, P)
                 : cudaLaunchKernelEx(&cfg, mk_megakernel, P);
}

cudaError_t launch_row_scale(uint8_t *dst, const uint8_t *src, const int32_t *map,
                             const uint64_t *scaletab, uint32_t nrows, uint32_t K,
                             cudaStream_t stream) {
  const uint32_t blocks = std::min<uint32_t>(65535u, (nrows + 7) / 8);
  mk_row_scale<<<blocks ? blocks : 1, 256, 0, stream>>>(dst, src, map, scaletab, nrows, K);
  return cudaGetLastError();
}

cudaError_t launch_retile_q8(uint8_t *dst, const uint8_t *src, const int32_t *map,
                             const uint64_t *rowtab, const uint64_t *scaletab, uint32_t nrows,
                             const OpGeom &g, uint32_t page, cudaStream_t stream) {
  const uint64_t total = (uint64_t)nrows * g.K / 8;
  const uint32_t blocks = (uint32_t)((total + 255) / 256 < 65535 ? (total + 255) / 256 : 65535);
  mk_retile_q8<<<blocks ? blocks : 1, 256, 0, stream>>>(dst, src, map, rowtab, scaletab, nrows,
                                                        g.K, g.NS, g.item_bytes, g.ipp, page);
  return cudaGetLastError();
}

cudaError_t launch_epoch_advance(uint32_t *ctrl, cudaStream_t stream) {
  mk_epoch_advance<<<1, 1, 0, stream>>>(ctrl);
  return cudaGetLastError();
}

cudaError_t launch_retile_tc(uint8_t *dst, const uint8_t *src, const int32_t *map,
                             uint32_t nrows, const OpGeom &g, uint32_t page, cudaStream_t stream) {
  const uint64_t total = (uint64_t)nrows * g.K / 8;
  const uint32_t blocks = (uint32_t)((total + 255) / 256 < 65535 ? (total + 255) / 256 : 65535);
  mk_retile_tc<<<blocks ? blocks : 1, 256, 0, stream>>>(dst, src, map, nrows, g.K, g.MR, g.kc,
                                                         g.kp, page);
  return cudaGetLastError();
}

cudaError_t launch_retile(uint8_t *dst, const uint8_t *src, const int32_t *map,
                          const uint64_t *rowtab, uint32_t nrows, const OpGeom &g, uint32_t page,
                          cudaStream_t stream) {
  const uint64_t total = (uint64_t)nrows * g.K * 2 / 16;
  const uint32_t blocks = (uint32_t)((total + 255) / 256 < 65535 ? (total + 255) / 256 : 65535);
  mk_retile<<<blocks ? blocks : 1, 256, 0, stream>>>(dst, src, map, rowtab, nrows, g.K, g.NS,
                                                      g.item_bytes, g.ipp, page);
  return cudaGetLastError();
}

}  // namespace mk
