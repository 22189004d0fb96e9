// mk_stream.cu -- the batch-1 persistent decode megakernel in which every
// compute warp streams its own weights (sm_103a).
//
// Same interpreter, instruction table and dependency counters as the shared
// page ring of mk_kernel.cu (« 2 · Définition et généalogie », §2.1 and §2.6),
// with the producer/consumer split of « 5 · La spécialisation des warps »
// (§5.2, §5.4) placed differently:
//   warp 0       publisher and dependency poller: claims instructions into
//                the FIFO, polls each instruction's input counter (acquire)
//                and, for the normalised projections and the O projection,
//                stages the input vector in shared memory (x / rms times the
//                gains, or the attention output) before releasing the slot's
//                ready barrier.
//   warp 1       storer: epilogues (RoPE and KV append, residual add,
//                SiLU(gate) * up, logits), the release of the instruction's
//                counter, the attention arrival and the group merge.
//   warps 2..15  compute: each warp streams ITS share of every tile (and, in
//                an attention chunk, its share of the key and value rows)
//                through a private ring of 512-byte slots filled by per-lane
//                async copies (cp.async), running ahead across instruction
//                boundaries and dependency waits (§5.4: the next op's weights
//                load while the current one finishes).
// Why not the shared page ring here: on sm_103a a gpu-scope release waits for
// the SM's bulk (TMA) copies in flight, so with a ring of bulk copies every
// hand-off between instructions costs several microseconds; per-lane async
// copies in flight in other warps do not hold the storer's release up, and
// the two warps that release or acquire never have copies of their own in
// flight.
#include "mk_device.cuh"

namespace mk {

constexpr uint32_t kWhereStream = 6u << 28;  // a ring wait found its slot never issued

// ------------------------------------------------------------- cp.async ----
DEVI void cp_async16(void *dst, const void *src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(saddr(dst)), "l"(src) : "memory");
}
DEVI void cp_async16_s(uint32_t dst, const void *src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}
// one commit group's four slots: 16 bytes each at dst + 512 t from src + 512 t
DEVI void cp_async16x4(uint32_t dst, const void *src) {
  asm volatile(
      "cp.async.cg.shared.global [%0], [%1], 16;\n\t"
      "cp.async.cg.shared.global [%0+512], [%1+512], 16;\n\t"
      "cp.async.cg.shared.global [%0+1024], [%1+1024], 16;\n\t"
      "cp.async.cg.shared.global [%0+1536], [%1+1536], 16;" ::"r"(dst),
      "l"(src)
      : "memory");
}
DEVI void cp_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
// 16-byte load from a shared-window address (an explicit shared-space load,
// never a generic one)
DEVI uint4 lds128(uint32_t a) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "r"(a) : "memory");
  return v;
}
DEVI uint32_t lds32(uint32_t a) {
  uint32_t v;
  asm volatile("ld.shared.u32 %0, [%1];" : "=r"(v) : "r"(a) : "memory");
  return v;
}
DEVI uint2 lds64(uint32_t a) {
  uint2 v;
  asm volatile("ld.shared.v2.u32 {%0,%1}, [%2];" : "=r"(v.x), "=r"(v.y) : "r"(a) : "memory");
  return v;
}
DEVI void cp_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }
// wait until at most n of this thread's most recent commit groups are pending
// (n < 8: the rings hold at most kMaxWarpRing / kSG groups)
DEVI void cp_wait_pending(uint32_t n) {
  switch (n) {
    case 0: asm volatile("cp.async.wait_group 0;" ::: "memory"); break;
    case 1: asm volatile("cp.async.wait_group 1;" ::: "memory"); break;
    case 2: asm volatile("cp.async.wait_group 2;" ::: "memory"); break;
    case 3: asm volatile("cp.async.wait_group 3;" ::: "memory"); break;
    case 4: asm volatile("cp.async.wait_group 4;" ::: "memory"); break;
    case 5: asm volatile("cp.async.wait_group 5;" ::: "memory"); break;
    case 6: asm volatile("cp.async.wait_group 6;" ::: "memory"); break;
    default: asm volatile("cp.async.wait_group 7;" ::: "memory"); break;
  }
}

// ------------------------------------------------------- a warp's stream ----
// The bytes one compute warp reads for one instruction: at most two
// contiguous ranges of global memory (a GEMV tile: the warp's run of items;
// an attention chunk: its key rows, then the same value rows).  In the ring a
// range occupies consecutive 512-byte slots, lane l copying (and, in a GEMV,
// reading) bytes [16 l, 16 l + 16) of each slot; an instruction's slots are
// padded to whole commit groups.
struct Ranges {
  const uint8_t *b0, *b1;
  uint32_t n0, n1;  // bytes
  uint32_t c0;      // slots of range 0 (range 1 follows it)
  uint32_t ctot;    // slots of the instruction, a multiple of kSG
};

// Items of a GEMV tile are stored in (slice, row) order; warp cw takes the
// contiguous run [a, b) of them.
DEVI void gemv_share(const KParams &P, const mk_instr &in, int cw, uint32_t &a, uint32_t &b,
                     uint32_t &wrows) {
  const OpGeom &G = P.geom[in.op];
  wrows = in.op == MK_OP_GATEUP ? 2 * in.nrows : in.nrows;
  const uint32_t n = wrows * G.NS;
  a = (uint32_t)cw * n / kComputeWarps;
  b = (uint32_t)(cw + 1) * n / kComputeWarps;
}

// Rows [j0, j1) of the chunk's n_tot positions served by warp cw (its head
// is cw % QPG); rows below n_old come from the cache, row n_old (the current
// position) from this step's key and value.
DEVI void attn_share(const KParams &P, const Smem &S, const mk_instr &in, int cw, int &p0,
                     int &n_tot, int &n_old, int &j0, int &j1) {
  const int pos = S.pos[in.b];
  int p1;
  attn_range(P, pos, in.chunk, p0, p1);
  n_tot = p1 - p0;
  n_old = max(0, min(p1, pos) - p0);
  const int QPG = P.qpg, h = cw % QPG, r = cw / QPG;
  const int nqs = (kComputeWarps - 1 - h) / QPG + 1;  // warps serving head h
  const int len = (max(n_tot, 0) + nqs - 1) / nqs;
  j0 = min(r * len, max(n_tot, 0));
  j1 = min(j0 + len, max(n_tot, 0));
}

DEVI void warp_ranges(const KParams &P, const Smem &S, const mk_instr &in, int cw, Ranges &R) {
  R.b0 = R.b1 = nullptr;
  R.n0 = R.n1 = 0;
  if (in.op != MK_OP_ATTN) {
    uint32_t a, b, wrows;
    gemv_share(P, in, cw, a, b, wrows);
    const uint32_t ib = P.geom[in.op].item_bytes;
    R.b0 = P.arena + in.wofs + (uint64_t)a * ib;
    R.n0 = (b - a) * ib;
  } else {
    int p0, n_tot, n_old, j0, j1;
    attn_share(P, S, in, cw, p0, n_tot, n_old, j0, j1);
    const int rows = max(0, min(j1, n_old) - j0);
    if (rows > 0) {
      const size_t at = kv_row(P, in.layer, in.b, in.g, p0 + j0);
      R.b0 = reinterpret_cast<const uint8_t *>(P.kc + at);
      R.b1 = reinterpret_cast<const uint8_t *>(P.vc + at);
      R.n0 = R.n1 = (uint32_t)rows * (uint32_t)P.d * 2u;
    }
  }
  R.c0 = (R.n0 + 511u) / 512u;
  R.ctot = (R.c0 + (R.n1 + 511u) / 512u + kSG - 1) / kSG * kSG;
}

// A compute warp's ring and its two cursors (values uniform across lanes,
// except the per-lane source pointers).
struct WStream {
  uint32_t ring;     // shared-window address of slot 0 of this warp's ring, plus 16 * lane
  uint32_t nb;       // slots
  uint32_t iss;      // positions issued (a multiple of kSG); position p sits in slot p % nb
  uint32_t islot;    // slot of position iss
  uint32_t con;      // positions the consumer is done with
  uint32_t cslot;    // slot of position con
  uint32_t fi;       // FIFO entry of the issue cursor
  uint32_t gl;       // commit groups of entry fi still to issue
  uint32_t state;    // 0: entry fi not examined yet, 1: issuing entry fi, 2: END reached
  int32_t r0, r1;    // bytes of range 0 / range 1 from the next slot on (<= 0: none left)
  const uint8_t *p0, *p1;  // this lane's next source bytes in range 0 / range 1
};

DEVI uint32_t slot_add(uint32_t slot, uint32_t n, uint32_t nb) {  // n <= nb
  slot += n;
  return slot >= nb ? slot - nb : slot;
}

// Issue commit groups while the ring has room and the cursor's FIFO entries
// are published.  Only published entries are read: every entry before them
// was published earlier, so a slot's parity test is never a round behind.
// An entry's slots: range 0, then range 1, then padding to a whole group.
DEVI void issue_more(const KParams &P, const Smem &S, WStream &W, int cw, int lane) {
  while (W.state != 2u && W.iss + kSG <= W.con + W.nb) {
    if (W.state == 0u) {
      const uint32_t f = W.fi % kFifo;
      const int pub = __shfl_sync(0xFFFFFFFFu, mbar_test(&S.ifull[f], (W.fi / kFifo) & 1u), 0);
      if (!pub) return;
      if (S.fifo[f].op == MK_OP_END) {
        W.state = 2u;
        return;
      }
      Ranges R;
      warp_ranges(P, S, S.fifo[f], cw, R);
      if (R.ctot == 0) {  // nothing of this entry for this warp
        ++W.fi;
        continue;
      }
      W.p0 = R.b0 + lane * 16;
      W.p1 = R.b1 + lane * 16;
      W.r0 = (int32_t)R.n0;
      W.r1 = (int32_t)R.n1;
      W.gl = R.ctot / kSG;
      W.state = 1u;
    }
    if (W.r0 >= (int32_t)(kSG * 512)) {  // a whole group of range 0 (the common case)
      cp_async16x4(W.ring + W.islot * 512u, W.p0);
      W.p0 += kSG * 512;
      W.r0 -= kSG * 512;
      W.islot = W.islot + kSG == W.nb ? 0u : W.islot + kSG;
      cp_commit();
      W.iss += kSG;
      if (--W.gl == 0u) {
        ++W.fi;
        W.state = 0u;
      }
      continue;
    }
    const int32_t me = lane * 16;
#pragma unroll
    for (int t = 0; t < kSG; ++t) {
      const uint32_t dst = W.ring + W.islot * 512u;
      if (W.r0 > 0) {
        if (me < W.r0) cp_async16_s(dst, W.p0);
        W.p0 += 512;
        W.r0 -= 512;
      } else if (W.r1 > 0) {
        if (me < W.r1) cp_async16_s(dst, W.p1);
        W.p1 += 512;
        W.r1 -= 512;
      }
      W.islot = W.islot + 1u == W.nb ? 0u : W.islot + 1u;
    }
    cp_commit();
    W.iss += kSG;
    if (--W.gl == 0u) {
      ++W.fi;
      W.state = 0u;
    }
  }
}

// Every lane waits for its own copies of positions <= c (issued earlier).
DEVI bool wait_upto(const KParams &P, const Smem &S, WStream &W, uint32_t c, int cw, int lane) {
  issue_more(P, S, W, cw, lane);
  if (c >= W.iss) {  // cannot happen by construction; never wait for a slot not issued
    if (lane == 0) {
      raise_error(P, MK_ERR_TIMEOUT, kWhereStream | (uint32_t)cw, true);
      S.misc[0] = 1;
    }
    return false;
  }
  cp_wait_pending(W.iss / kSG - c / kSG - 1u);
  return true;
}

// ------------------------------------------------------------------ GEMV ----
// The dot product runs on packed pairs of fp32 (fma.rn.f32x2): the two bf16
// of a weight word, widened exactly, times two consecutive inputs.
struct XPack {
  unsigned long long p[kSG][4];  // chunk j, pair m: inputs (8 m' + 2 m, + 1) of the lane's slice
};
DEVI unsigned long long pack2(float a, float b) {
  unsigned long long r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(a), "f"(b));
  return r;
}
DEVI float sum2(unsigned long long v) {
  float a, b;
  asm("mov.b64 {%0, %1}, %2;" : "=f"(a), "=f"(b) : "l"(v));
  return a + b;
}
// acc += (lo bf16 of w, hi bf16 of w) * (x0, x1), elementwise in fp32
DEVI void fma_bf2(unsigned long long &acc, uint32_t w, unsigned long long xp) {
  asm("{\n\t.reg .b32 lo, hi;\n\t.reg .b64 wp;\n\t"
      "shl.b32 lo, %1, 16;\n\tand.b32 hi, %1, 0xFFFF0000;\n\t"
      "mov.b64 wp, {lo, hi};\n\tfma.rn.f32x2 %0, wp, %2, %0;\n\t}"
      : "+l"(acc)
      : "r"(w), "l"(xp));
}
DEVI void load_x_pack(const KParams &P, const Smem &S, int op, uint32_t s, int lane, float r,
                      XPack &X) {
  const OpGeom &G = P.geom[op];
#pragma unroll
  for (int j = 0; j < kSG; ++j) {
    if ((uint32_t)j >= G.nch) break;
    const uint32_t col = s * G.SW + (uint32_t)j * 256u + (uint32_t)lane * 8u;
    float4 a, c;
    if (op == MK_OP_DOWN) {
      a = __ldcg(reinterpret_cast<const float4 *>(P.h + col));
      c = __ldcg(reinterpret_cast<const float4 *>(P.h + col + 4));
    } else {
      const uint32_t xa = saddr(S.xs + col);
      const uint4 ua = lds128(xa), uc = lds128(xa + 16);
      a = make_float4(__uint_as_float(ua.x) * r, __uint_as_float(ua.y) * r,
                      __uint_as_float(ua.z) * r, __uint_as_float(ua.w) * r);
      c = make_float4(__uint_as_float(uc.x) * r, __uint_as_float(uc.y) * r,
                      __uint_as_float(uc.z) * r, __uint_as_float(uc.w) * r);
    }
    X.p[j][0] = pack2(a.x, a.y);
    X.p[j][1] = pack2(a.z, a.w);
    X.p[j][2] = pack2(c.x, c.y);
    X.p[j][3] = pack2(c.z, c.w);
  }
}
// one item: nch (<= kSG) consecutive slots from ring byte `soff` on (advanced
// past them), this lane's 16 bytes of each
DEVI float dot_item(uint32_t ring, uint32_t &soff, uint32_t rbytes, uint32_t nch,
                    const XPack &X) {
  unsigned long long A = 0ull, B = 0ull;  // packed (+0, +0)
#pragma unroll
  for (int j = 0; j < kSG; ++j)
    if ((uint32_t)j < nch) {
      const uint4 w = lds128(ring + soff);
      fma_bf2(A, w.x, X.p[j][0]);
      fma_bf2(B, w.y, X.p[j][1]);
      fma_bf2(A, w.z, X.p[j][2]);
      fma_bf2(B, w.w, X.p[j][3]);
      soff = soff + 512u == rbytes ? 0u : soff + 512u;
    }
  return sum2(A) + sum2(B);
}

// Stage the input of a normalised projection (x, or the embedding row of the
// layer-0 token, times the gains) or of the O projection (the attention
// output) into xs, every compute thread four columns at a time, with each
// warp's sum of squares of x at xs[K + warp]; then a compute-warp barrier.
// Once per change of input: the next instruction with another input depends
// (through the counters) on every instruction of this one, this block's
// included, so no warp still reads xs when it is restaged.
DEVI bool stage_input_stream(const KParams &P, const Smem &S, const mk_instr &in, int cw, int lane,
                             uint32_t &xbar_uses) {
  const uint32_t K = P.geom[in.op].K;
  float *xs = S.xs;
  const bool oproj = in.op == MK_OP_OPROJ;
  const uint16_t *gain = gain_of(P, in.op, in.layer);
  const int emb = in.op == MK_OP_QKV && (in.flags & 1);
  const uint16_t *erow = P.embed + (size_t)S.tok[0] * P.H;
  float ss = 0.f;
  for (uint32_t i = ((uint32_t)cw * 32u + (uint32_t)lane) * 4u; i < K; i += kComputeWarps * 128u) {
    float4 v;
    if (oproj) {
      v = __ldcg(reinterpret_cast<const float4 *>(P.attn + i));
    } else {
      if (emb) {
        const uint2 e = __ldg(reinterpret_cast<const uint2 *>(erow + i));
        v = make_float4(bf_lo(e.x), bf_hi(e.x), bf_lo(e.y), bf_hi(e.y));
      } else {
        v = __ldcg(reinterpret_cast<const float4 *>(P.x + i));
      }
      const uint2 g = __ldg(reinterpret_cast<const uint2 *>(gain + i));
      ss = fmaf(v.x, v.x, fmaf(v.y, v.y, fmaf(v.z, v.z, fmaf(v.w, v.w, ss))));
      v = make_float4(v.x * bf_lo(g.x), v.y * bf_hi(g.x), v.z * bf_lo(g.y), v.w * bf_hi(g.y));
    }
    *reinterpret_cast<float4 *>(xs + i) = v;
  }
  ss = warp_sum(ss);
  if (lane == 0) xs[K + cw] = ss;
  return compute_sync(P, S, S.xbar, xbar_uses, lane);
}

// The warp's run of items of one tile, two at a time where they share a
// slice; item (row r, slice s) leaves its dot product in res[r NS + s].
DEVI bool gemv_stream(const KParams &P, const Smem &S, const mk_instr &in, const SlotMeta &meta,
                      float *res, int cw, int lane, WStream &W) {
  const OpGeom &G = P.geom[in.op];
  uint32_t a, b, wrows;
  gemv_share(P, in, cw, a, b, wrows);
  const uint32_t epos = W.con, nch = G.nch;
  uint32_t xs_ = 0xFFFFFFFFu;  // slice whose inputs are in Xp
  // 1/rms of a normalised input, from the staging warps' sums of squares
  float r = 1.f;
  if (gain_of(P, in.op, in.layer) != nullptr) {
    float ss = 0.f;
    for (int w = 0; w < kComputeWarps; ++w) ss += S.xs[G.K + w];
    r = rsqrtf(ss / (float)G.K + P.eps);
  }
  const bool stamp = cw == 0 && lane == 0 && (P.flags & MK_FLAG_TRACE);
  SlotMeta &mw = const_cast<SlotMeta &>(meta);  // meta is this entry's slot in shared memory
  // Items two at a time where they share a slice; the two sums reduced
  // together (lanes 0..15 end with the first, 16..31 with the second).
  XPack Xp;
  uint32_t s = a / wrows, rr = a - s * wrows;
  uint32_t soff = W.cslot * 512u;  // ring byte of the next item's first slot (this lane's part)
  const uint32_t rbytes = W.nb * 512u;
  for (uint32_t i = a; i < b;) {
    if (s != xs_) {
      load_x_pack(P, S, in.op, s, lane, r, Xp);
      xs_ = s;
    }
    if (stamp && i == a) mw.t_input = gtimer();
    const bool two = i + 1 < b && rr + 1 < wrows;
    const uint32_t cl = W.con + (two ? 2u : 1u) * nch - 1u;
    if (!wait_upto(P, S, W, cl, cw, lane)) return false;
    if (stamp && i == a) mw.t_page0 = gtimer();
    const float acc = dot_item(W.ring, soff, rbytes, nch, Xp);
    const float acc2 = two ? dot_item(W.ring, soff, rbytes, nch, Xp) : 0.f;
    const bool up = (lane & 16) != 0;
    float v = (up ? acc2 : acc) + __shfl_xor_sync(0xFFFFFFFFu, up ? acc : acc2, 16);
#pragma unroll
    for (int o = 8; o; o >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, o);
    if (lane == 0) res[rr * G.NS + s] = v;
    if (two && lane == 16) res[(rr + 1) * G.NS + s] = v;
    W.con = cl + 1u;
    const uint32_t n = two ? 2u : 1u;
    i += n;
    rr += n;
    if (rr >= wrows) {
      rr -= wrows;
      ++s;
    }
  }
  if (stamp) mw.t_pagel = gtimer();
  // skip the instruction's padding slots; refill the ring
  const uint32_t ctot = ((b - a) * nch + kSG - 1) / kSG * kSG;
  W.cslot = slot_add(soff / 512u, epos + ctot - W.con, W.nb);
  W.con = epos + ctot;
  issue_more(P, S, W, cw, lane);
  return true;
}

// ------------------------------------------------------------- attention ----
// One split-KV chunk for the QPG query heads of group g of sequence b: the
// same computation as the shared-ring kernel's attention chunk (scores
// q.k / sqrt(d), the chunk's maximum m, denominator l = sum exp(s - m),
// unnormalised o = sum exp(s - m) v, the per-warp partials merged per head
// in the block, the chunk partial {m[QPG], l[QPG], o[QPG][D]} written to
// global memory); the key and value rows below p_b come from the warp's own
// ring, the current position's from this step's key and value.  The
// arrival and the merge of the group are the storer's.
// The caller has waited for every slot of the entry (all lanes, then a warp
// barrier): ring0 is the warp's slot 0, slot0 the slot of the entry's first position.
template <int D, int QPG>
__device__ __noinline__ bool attn_stream(const KParams &P, const Smem &S, const mk_instr &in,
                                         const SlotMeta &meta, int cw, int lane, uint32_t att_uses,
                                         uint32_t ring0, uint32_t nb, uint32_t slot0) {
  constexpr int LPP = D / 8;      // lanes per key row (16 bytes each)
  constexpr int RPS = 32 / LPP;   // key rows per warp step
  constexpr int DPL = D / 32;     // value dims per lane
  const int b = in.b, g = in.g, pos = S.pos[b];
  int p0, n_tot, n_old, j0, j1;
  attn_share(P, S, in, cw, p0, n_tot, n_old, j0, j1);
  const int h = cw % QPG;
  const int part = lane % LPP;
  const bool stamp = cw == 0 && lane == 0 && (P.flags & MK_FLAG_TRACE);
  SlotMeta &mw = const_cast<SlotMeta &>(meta);  // this entry's slot in shared memory
  if (n_tot <= 0) return true;  // a chunk past p_b: nothing to do (the storer skips it too)
  Ranges R;
  warp_ranges(P, S, in, cw, R);
  const uint32_t rbytes = nb * 512u;
  const uint32_t kofs = slot0 * 512u;                       // ring byte of key row j0
  const uint32_t vofs = slot_add(slot0, R.c0, nb) * 512u;   // ring byte of value row j0
  auto krow = [&](int j) {  // shared address of key row j (j0 <= j < n_old) in the ring
    uint32_t o = kofs + (uint32_t)(j - j0) * (uint32_t)(D * 2);
    if (o >= rbytes) o -= rbytes;
    return ring0 + o;
  };
  auto vrow = [&](int j) {
    uint32_t o = vofs + (uint32_t)(j - j0) * (uint32_t)(D * 2);
    if (o >= rbytes) o -= rbytes;
    return ring0 + o;
  };

  // query slice of head h (8 dims per lane), pre-scaled by 1/sqrt(d); the
  // current position's key slice and value dims if this warp covers p_b
  float q8[8], kn8[8], vn[DPL];
  {
    const size_t qo = ((size_t)b * P.nq + (size_t)g * QPG + h) * D + part * 8;
    const float4 x0 = __ldcg(reinterpret_cast<const float4 *>(P.q + qo));
    const float4 x1 = __ldcg(reinterpret_cast<const float4 *>(P.q + qo + 4));
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

  // 1. scores of rows j0..j1 into this warp's row of S.sc (transposing
  //    butterfly over the LPP lanes of a row group)
  float *__restrict__ sw = S.sc + (size_t)cw * P.att_lmax;
  for (int jb = j0; jb < j1; jb += LPP * RPS) {
    float v[LPP];
#pragma unroll
    for (int t = 0; t < LPP; ++t) {
      const int j = jb + t * RPS + lane / LPP;
      float k8[8];
      if (j < n_old) {
        const uint4 w = lds128(krow(j) + part * 16);
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
  if (stamp) mw.t_pagel = gtimer();
  float o[8][DPL];
#pragma unroll
  for (int u = 0; u < 8; ++u)
#pragma unroll
    for (int k = 0; k < DPL; ++k) o[u][k] = 0.f;
  const int jo = min(j1, n_old);  // rows of this warp that come from the ring
  int j = j0;
  for (; j + 8 <= jo; j += 8) {
    const float4 pa = *reinterpret_cast<const float4 *>(sw + (j - j0));
    const float4 pb = *reinterpret_cast<const float4 *>(sw + (j - j0) + 4);
    const float pj[8] = {pa.x, pa.y, pa.z, pa.w, pb.x, pb.y, pb.z, pb.w};
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const uint32_t row = vrow(j + u) + lane * DPL * 2;
      if constexpr (DPL == 2) {
        const uint32_t w = lds32(row);
        o[u][0] = fmaf(pj[u], bf_lo(w), o[u][0]);
        o[u][1] = fmaf(pj[u], bf_hi(w), o[u][1]);
      } else {
        const uint2 w = lds64(row);
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
      const uint32_t row = vrow(j) + lane * DPL * 2;
#pragma unroll
      for (int k = 0; k < DPL; k += 2) {
        const uint32_t w = lds32(row + k * 2);
        o[0][k] = fmaf(pj, bf_lo(w), o[0][k]);
        o[0][k + 1] = fmaf(pj, bf_hi(w), o[0][k + 1]);
      }
    } else {
#pragma unroll
      for (int k = 0; k < DPL; ++k) o[0][k] = fmaf(pj, vn[k], o[0][k]);
    }
  }
  // the warp is done with its rows: every lane has read them before any lane
  // refills the slots (the caller refills after this returns)
  __syncwarp();

  // 4. per-warp partials (double-buffered by instruction parity)
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
  return true;
}

// Waits for every slot of the entry, runs the chunk, then releases the slots.
DEVI bool attn_stream_dispatch(const KParams &P, const Smem &S, const mk_instr &in,
                               const SlotMeta &meta, int cw, int lane, uint32_t &att_uses,
                               WStream &W) {
  Ranges R;
  warp_ranges(P, S, in, cw, R);
  const uint32_t epos = W.con;
  if (R.ctot) {
    // every lane waits for its own copies; the warp barrier then makes all
    // lanes' slots visible to every lane
    if (!wait_upto(P, S, W, epos + R.ctot - 1u, cw, lane)) return false;
    __syncwarp();
  }
  const uint32_t ring0 = W.ring - (uint32_t)lane * 16u;
  const uint32_t nb = W.nb, uses = att_uses, slot0 = W.cslot;
  bool ok;
  if (P.d == 64) {
    switch (P.qpg) {
      case 1: ok = attn_stream<64, 1>(P, S, in, meta, cw, lane, uses, ring0, nb, slot0); break;
      case 2: ok = attn_stream<64, 2>(P, S, in, meta, cw, lane, uses, ring0, nb, slot0); break;
      case 4: ok = attn_stream<64, 4>(P, S, in, meta, cw, lane, uses, ring0, nb, slot0); break;
      default: ok = attn_stream<64, 8>(P, S, in, meta, cw, lane, uses, ring0, nb, slot0); break;
    }
  } else {
    switch (P.qpg) {
      case 1: ok = attn_stream<128, 1>(P, S, in, meta, cw, lane, uses, ring0, nb, slot0); break;
      case 2: ok = attn_stream<128, 2>(P, S, in, meta, cw, lane, uses, ring0, nb, slot0); break;
      case 4: ok = attn_stream<128, 4>(P, S, in, meta, cw, lane, uses, ring0, nb, slot0); break;
      default: ok = attn_stream<128, 8>(P, S, in, meta, cw, lane, uses, ring0, nb, slot0); break;
    }
  }
  // a chunk with work passes one compute-warp barrier (the per-warp merge)
  if (ok && (int)(S.pos[in.b] - (int)in.chunk * P.attn_chunk) >= 0) ++att_uses;
  W.con = epos + R.ctot;
  W.cslot = slot_add(W.cslot, R.ctot, W.nb);
  issue_more(P, S, W, cw, lane);
  return ok;
}

// --------------------------------------------------------- compute warps ----
DEVI void compute_stream(const KParams &P, const Smem &S, int cw, int lane) {
  WStream W;
  W.ring = saddr(S.wring) + (uint32_t)cw * P.wnb * 512u + (uint32_t)lane * 16u;
  W.nb = P.wnb;
  W.iss = W.islot = W.con = W.cslot = W.fi = W.gl = W.state = 0u;
  W.r0 = W.r1 = 0;
  W.p0 = W.p1 = nullptr;
  uint32_t att_uses = 0, xbar_uses = 0, skey = 0xFFFFFFFFu;
  for (uint32_t fs = 0;; ++fs) {
    if (!next_entry(P, S, fs)) break;
    issue_more(P, S, W, cw, lane);  // the new entry's slots go out before its dependency wait
    const uint32_t f = fs % kFifo;
    const mk_instr &in = S.fifo[f];
    const SlotMeta &meta = S.meta[f];
    if (in.op == MK_OP_END) {
      finish_entry(P, S, fs, cw, lane);
      break;
    }
    if (!warp_wait(P, S, &S.rdy[f], (fs / kFifo) & 1u, kWhereCompute | meta.idx)) break;
    bool ok;
    if (in.op == MK_OP_ATTN) {
      ok = attn_stream_dispatch(P, S, in, meta, cw, lane, att_uses, W);
    } else {
      if (in.op != MK_OP_DOWN && input_key(in) != skey) {
        if (!stage_input_stream(P, S, in, cw, lane, xbar_uses)) break;
        skey = input_key(in);
      }
      ok = gemv_stream(P, S, in, meta, S.res + (size_t)f * P.res_floats, cw, lane, W);
    }
    if (!ok) break;
    finish_entry(P, S, fs, cw, lane);
  }
  cp_wait_all();  // no copy of this warp's may land after the block exits
}

// ------------------------------------------------ publisher and poller ----
DEVI void load_record(const KParams &P, uint32_t idx, uint4 (&r)[4]) {
  if (idx < P.n_instr) {
    const uint4 *src = reinterpret_cast<const uint4 *>(P.instr + idx);
#pragma unroll
    for (int i = 0; i < 4; ++i) r[i] = __ldg(src + i);
  }
}

// One poll of an instruction's input counter (no wait): true once this
// step's target is reached.  `sat` caches satisfied targets for the launch.
DEVI bool poll_once(const KParams &P, const Smem &S, const mk_instr &in, uint32_t epoch) {
  if (P.mode == kModeRange || in.wait_ctr == MK_NO_COUNTER) return true;
  const uint32_t c = in.wait_ctr;
  const uint32_t target = epoch * __ldg(P.ctr_inc + c) + in.wait_tgt;
  const bool cacheable = c < (uint32_t)P.n_wait;
  if (cacheable && S.sat[c] != 0 && (int32_t)((S.sat[c] - 1u) - target) >= 0) return true;
  if ((int32_t)(ld_acquire(P.ctr + (size_t)c * kCtrStride) - target) < 0) return false;
  if (cacheable) S.sat[c] = target + 1u;
  return true;
}

// Warp 0: publishes instructions into the FIFO as slots free up (lane 0:
// queue claim, list entry or range, two claims and records ahead), and makes
// published entries ready in order: polls the input counter, then releases
// the slot's ready barrier.  Neither job waits on the other: a counter not
// yet reached is polled again after the next publish.
DEVI void poller_stream(const KParams &P, const Smem &S, uint32_t epoch, int lane) {
  const uint32_t N = P.n_instr;
  const uint32_t qbase = epoch * (N + P.n_blocks);
  uint32_t list_k = 0, list_end = 0, range_taken = 0;
  if (P.mode == kModeStatic) {
    list_k = P.list_off[blockIdx.x];
    list_end = P.list_off[blockIdx.x + 1];
  }
  auto claim = [&]() -> uint32_t {  // lane 0 only
    if (P.mode == kModeDynamic) return atomicAdd(P.ctrl + kCtlQueue, 1u) - qbase;
    if (P.mode == kModeStatic) return list_k < list_end ? __ldg(P.list_idx + list_k++) : N;
    const uint32_t r = range_taken ? N : P.range_first + blockIdx.x;
    range_taken = 1;
    return r;
  };
  uint4 ra[4], rb[4];
  uint32_t a = N, b = N, c = N;
  if (lane == 0) {
    a = claim();
    load_record(P, a, ra);
    if (a < N) b = claim();
    load_record(P, b, rb);
    if (b < N) c = claim();
  }
  uint32_t fs_c = 0, fs_p = 0;  // entries published, entries made ready
  uint32_t ended = 0;           // END published
  uint64_t t_idle = 0;
  uint32_t n_idle = 0;
  while (true) {
    bool progress = false;
    // ---- publish (lane 0)
    int pub = 0;
    if (lane == 0 && !ended && fs_c - fs_p < P.lookahead) {
      const uint32_t f = fs_c % kFifo, k = fs_c / kFifo;
      if (k == 0 || mbar_test(&S.iempty[f], (k - 1) & 1u)) {
        if (a >= N) {
          S.fifo[f].op = MK_OP_END;
          S.meta[f].idx = N;
          S.meta[f].npages = 0;
          mbar_arrive(&S.ifull[f]);
          ended = 1;
        } else {
          uint4 *dst = reinterpret_cast<uint4 *>(&S.fifo[f]);
#pragma unroll
          for (int i = 0; i < 4; ++i) dst[i] = ra[i];
          SlotMeta &m = S.meta[f];
          m.idx = a;
          m.seq0 = 0;
          m.npages = 0;
          m.t_claim = (P.flags & MK_FLAG_TRACE) ? gtimer() : 0ull;
          mbar_arrive(&S.ifull[f]);
          a = b;
#pragma unroll
          for (int i = 0; i < 4; ++i) ra[i] = rb[i];
          b = c;
          load_record(P, b, rb);
          c = b < N ? claim() : N;
        }
        pub = 1;
      }
    }
    pub = __shfl_sync(0xFFFFFFFFu, pub, 0);
    if (pub) {
      ++fs_c;
      progress = true;
    }
    ended = __shfl_sync(0xFFFFFFFFu, ended, 0);
    // ---- make entry fs_p ready
    if (fs_p < fs_c) {
      const uint32_t f = fs_p % kFifo;
      const mk_instr &in = S.fifo[f];
      if (in.op == MK_OP_END) break;  // the compute warps and the storer stop at END
      int ready = 0;
      if (lane == 0) ready = poll_once(P, S, in, epoch);
      ready = __shfl_sync(0xFFFFFFFFu, ready, 0);
      if (ready) {
        if (lane == 0) {
          if (P.flags & MK_FLAG_TRACE) S.meta[f].t_ready = gtimer();
          mbar_arrive(&S.rdy[f]);
        }
        ++fs_p;
        progress = true;
      }
    }
    if (progress) {
      t_idle = 0;
      n_idle = 0;
    } else {
      if (!t_idle) t_idle = cycles() | 1u;
      __nanosleep(32);
      int stop = 0;
      if (lane == 0) stop = should_stop(P, S, t_idle, n_idle, kWherePoll | fs_p);
      if (__shfl_sync(0xFFFFFFFFu, stop, 0)) break;
    }
  }
}

// --------------------------------------------------------------- storer ----
// Arrival of a finished attention chunk on its (sequence, group) counter;
// the chunk that completes the group merges the group's chunk partials by
// log-sum-exp, in chunk order, into the attention output and releases the
// group counter.  Chunks past p_b do not arrive: the last real chunk adds
// their share, so the counter advances by nchunk per step.  Lane l merges
// OPL consecutive outputs of one head, CB chunks' loads in flight.
template <int D, int QPG>
__device__ __noinline__ void storer_attn(const KParams &P, const Smem &S, const mk_instr &in,
                                         int lane, uint32_t epoch) {
  const int b = in.b, g = in.g, pos = S.pos[b];
  int p0, p1;
  attn_range(P, pos, in.chunk, p0, p1);
  if (p1 - p0 <= 0) return;
  const int nch = min((int)in.nchunk, (pos + P.attn_chunk) / P.attn_chunk);
  int last = 0;
  if (lane == 0) {
    uint32_t *ctr = P.ctr + (size_t)in.sig_ctr * kCtrStride;
    const uint32_t old = atom_add_acq_rel(ctr, 1u);
    last = old == epoch * in.nchunk + (uint32_t)nch - 1u;
    if (last && (uint32_t)nch < in.nchunk) red_add(ctr, in.nchunk - (uint32_t)nch);
  }
  if (!__shfl_sync(0xFFFFFFFFu, last, 0)) return;
  constexpr int OPL = QPG * D / 32;  // outputs per lane
  constexpr int CB0 = 80 / (OPL + 2);
  constexpr int CB = CB0 < 1 ? 1 : (CB0 > 16 ? 16 : CB0);
  const int o0 = lane * OPL, h = o0 / D;
  const int PS = 2 * QPG + QPG * D;
  const float *pb = P.part + ((size_t)b * P.nkv + g) * in.nchunk * PS;
  float M = -INFINITY, den = 0.f, num[OPL];
#pragma unroll
  for (int k = 0; k < OPL; ++k) num[k] = 0.f;
  for (int cb = 0; cb < nch; cb += CB) {
    float mc[CB], lc[CB], oc[CB][OPL];
#pragma unroll
    for (int u = 0; u < CB; ++u) {
      mc[u] = -INFINITY;
      lc[u] = 0.f;
#pragma unroll
      for (int k = 0; k < OPL; ++k) oc[u][k] = 0.f;
      if (cb + u < nch) {
        const float *pc = pb + (size_t)(cb + u) * PS;
        mc[u] = __ldcg(pc + h);
        lc[u] = __ldcg(pc + QPG + h);
        if constexpr (OPL % 4 == 0) {
#pragma unroll
          for (int k = 0; k < OPL; k += 4) {
            const float4 t = __ldcg(reinterpret_cast<const float4 *>(pc + 2 * QPG + o0 + k));
            oc[u][k] = t.x; oc[u][k + 1] = t.y; oc[u][k + 2] = t.z; oc[u][k + 3] = t.w;
          }
        } else {
#pragma unroll
          for (int k = 0; k < OPL; ++k) oc[u][k] = __ldcg(pc + 2 * QPG + o0 + k);
        }
      }
    }
#pragma unroll
    for (int u = 0; u < CB; ++u) {
      if (mc[u] == -INFINITY) continue;
      const float Mn = fmaxf(M, mc[u]);
      const float sa = __expf(M - Mn), sw = __expf(mc[u] - Mn);
      den = den * sa + sw * lc[u];
#pragma unroll
      for (int k = 0; k < OPL; ++k) num[k] = num[k] * sa + sw * oc[u][k];
      M = Mn;
    }
  }
  float *dst = P.attn + (size_t)b * P.nq * D + (size_t)g * QPG * D + o0;
#pragma unroll
  for (int k = 0; k < OPL; ++k) dst[k] = num[k] / den;
  __syncwarp();  // every lane's outputs before lane 0's release
  if (lane == 0) red_release(P.ctr + (size_t)in.sig2_ctr * kCtrStride, 1u);
}

DEVI void storer_attn_dispatch(const KParams &P, const Smem &S, const mk_instr &in, int lane,
                               uint32_t epoch) {
  if (P.d == 64) {
    switch (P.qpg) {
      case 1: storer_attn<64, 1>(P, S, in, lane, epoch); return;
      case 2: storer_attn<64, 2>(P, S, in, lane, epoch); return;
      case 4: storer_attn<64, 4>(P, S, in, lane, epoch); return;
      default: storer_attn<64, 8>(P, S, in, lane, epoch); return;
    }
  }
  switch (P.qpg) {
    case 1: storer_attn<128, 1>(P, S, in, lane, epoch); return;
    case 2: storer_attn<128, 2>(P, S, in, lane, epoch); return;
    case 4: storer_attn<128, 4>(P, S, in, lane, epoch); return;
    default: storer_attn<128, 8>(P, S, in, lane, epoch); return;
  }
}

DEVI void storer_stream(const KParams &P, const Smem &S, uint32_t epoch, int lane) {
  for (uint32_t fs = 0;; ++fs) {
    const uint32_t f = fs % kFifo, k = fs / kFifo;
    if (!warp_wait(P, S, &S.ifull[f], k & 1u, kWhereStorer)) break;
    const mk_instr &in = S.fifo[f];
    const SlotMeta &meta = S.meta[f];
    if (in.op == MK_OP_END) break;
    if (!warp_wait(P, S, &S.rdy[f], k & 1u, kWhereStorer)) break;
    prefetch_residual(P, S, in, lane);
    if (!warp_wait(P, S, &S.done[f], k & 1u, kWhereStorer)) break;
    if (lane == 0 && (P.flags & MK_FLAG_TRACE)) S.meta[f].t_sstart = gtimer();
    __syncwarp();
    if (in.op == MK_OP_ATTN) storer_attn_dispatch(P, S, in, lane, epoch);
    storer_epilogue(P, S, in, meta, S.res + (size_t)f * P.res_floats, lane, epoch);
    __syncwarp();
    if (lane == 0) mbar_arrive(&S.iempty[f]);
  }
}

// --------------------------------------------------------------- kernel ----
extern "C" __global__ void __launch_bounds__(kThreads, 1)
    mk_megakernel_stream(const __grid_constant__ KParams P) {
  extern __shared__ __align__(1024) uint8_t smem[];
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  Smem *desc = reinterpret_cast<Smem *>(smem + P.off_misc + kMiscDescOffset);
  if (tid == 0) *desc = make_smem(P, smem);
  __syncthreads();
  const Smem &S = *desc;
  if (tid == 0) {
    for (int i = 0; i < kFifo; ++i) {
      mbar_init(&S.ifull[i], 1);
      mbar_init(&S.iempty[i], 1);
      mbar_init(&S.rdy[i], 1);
      mbar_init(&S.done[i], kComputeWarps);
    }
    mbar_init(S.attbar, kComputeWarps);
    mbar_init(S.xbar, kComputeWarps);
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
  if (warp == 0) {
    poller_stream(P, S, epoch, lane);
  } else if (warp == 1) {
    storer_stream(P, S, epoch, lane);
  } else {
    compute_stream(P, S, warp - 2, lane);
  }
  __syncthreads();
  // a block only bails after a latched error; never let it end silently
  if (tid == 0 && S.misc[0] != 0) raise_error(P, MK_ERR_TIMEOUT, 0x0FFFFFFFu, true);
  if (tid == 0 && P.mode != kModeRange && S.misc[0] == 0) {
    fence_gpu();
    const uint32_t old = atomicAdd(P.ctrl + kCtlExit, 1u);
    if (old == epoch * P.n_blocks + P.n_blocks - 1u) atomicExch(P.ctrl + kCtlEpoch, epoch + 1u);
  }
}

// Re-tiling for stream plans: the 8 columns from c of arena row k (source
// row map[k], or k) go to item (row r, slice c / SW) of its tile, items in
// (slice, row) order: rowtab[k] = tile offset << 24 | tile rows << 12 | r.
extern "C" __global__ void mk_retile_stream(uint8_t *dst, const uint8_t *src, const int32_t *map,
                                            const uint64_t *rowtab, uint32_t nrows, uint32_t K,
                                            uint32_t SW) {
  const uint64_t per_row = K / 8;
  const uint64_t total = (uint64_t)nrows * per_row;
  for (uint64_t i = (uint64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total;
       i += (uint64_t)gridDim.x * blockDim.x) {
    const uint32_t k = (uint32_t)(i / per_row);
    const uint32_t c = (uint32_t)(i % per_row) * 8;
    const uint64_t rt = rowtab[k];
    const uint32_t r = (uint32_t)(rt & 4095u), rows = (uint32_t)((rt >> 12) & 4095u);
    const uint32_t s = c / SW, cc = c % SW;
    uint8_t *d = dst + (rt >> 24) + (((uint64_t)s * rows + r) * SW + cc) * 2;
    const uint32_t srow = map ? (uint32_t)map[k] : k;
    *reinterpret_cast<uint4 *>(d) =
        *reinterpret_cast<const uint4 *>(src + (uint64_t)srow * K * 2 + (uint64_t)c * 2);
  }
}

// ---- host-side launch helpers ----
cudaError_t set_stream_smem(uint32_t bytes) {
  return cudaFuncSetAttribute(mk_megakernel_stream, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              (int)bytes);
}

cudaError_t launch_megakernel_stream(const KParams &P, uint32_t grid, bool cooperative,
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
  return cudaLaunchKernelEx(&cfg, mk_megakernel_stream, P);
}

cudaError_t launch_retile_stream(uint8_t *dst, const uint8_t *src, const int32_t *map,
                                 const uint64_t *rowtab, uint32_t nrows, const OpGeom &g,
                                 cudaStream_t stream) {
  const uint64_t total = (uint64_t)nrows * g.K / 8;
  const uint32_t blocks = (uint32_t)((total + 255) / 256 < 65535 ? (total + 255) / 256 : 65535);
  mk_retile_stream<<<blocks ? blocks : 1, 256, 0, stream>>>(dst, src, map, rowtab, nrows, g.K,
                                                            g.SW);
  return cudaGetLastError();
}

}  // namespace mk
