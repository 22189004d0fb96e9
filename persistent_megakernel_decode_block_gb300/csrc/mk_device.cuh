// mk_device.cuh -- device helpers shared by the two translation units of the
// persistent decode megakernel: PTX wrappers (mbarriers, bulk copies, gpu-scope
// acquire/release), the shared-memory pointer table, bounded waits, the
// instruction FIFO hand-offs and the storer's epilogue.  Included by
// mk_kernel.cu (shared page ring: batch-1 ring plans and tensor-core plans)
// and mk_stream.cu (batch-1 plans whose compute warps stream their own
// weights).
#pragma once
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include "mk_internal.h"

namespace mk {

#define DEVI __device__ __forceinline__

// ---------------------------------------------------------------- PTX ----
DEVI uint32_t saddr(const void *p) { return static_cast<uint32_t>(__cvta_generic_to_shared(p)); }

DEVI void mbar_init(uint64_t *b, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(saddr(b)), "r"(count) : "memory");
}
DEVI void mbar_arrive(uint64_t *b) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(saddr(b)) : "memory");
}
DEVI void mbar_arrive_expect_tx(uint64_t *b, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(saddr(b)), "r"(bytes)
               : "memory");
}
// Potentially blocking: the thread may be suspended (up to the hint, 20 us)
// until the phase completes, so a waiting warp does not take issue slots
// from the warps sharing its scheduler; false if the phase is still open.
DEVI bool mbar_try_wait(uint64_t *b, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(saddr(b)), "r"(parity), "r"(20000u)
      : "memory");
  return ok != 0;
}
// non-blocking test of a phase
DEVI bool mbar_test(uint64_t *b, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(saddr(b)), "r"(parity)
      : "memory");
  return ok != 0;
}
// bulk prefetch of global memory into L2 (no shared memory, no completion)
DEVI void bulk_prefetch_l2(const void *src, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(src), "r"(bytes) : "memory");
}
// ---- tcgen05 (5th-generation tensor cores, accumulator in tensor memory) ----
// Shared-memory matrix descriptor: start address, byte strides between 8-row
// x 16-byte core matrices along K (lbo) and along M/N (sbo), no swizzle.
DEVI uint64_t tc_desc(uint32_t saddr_bytes, uint32_t lbo, uint32_t sbo) {
  return (uint64_t)((saddr_bytes >> 4) & 0x3FFFu) | ((uint64_t)((lbo >> 4) & 0x3FFFu) << 16) |
         ((uint64_t)((sbo >> 4) & 0x3FFFu) << 32) | ((uint64_t)1 << 46);
}
// Instruction descriptor of kind::f16: fp32 accumulator, bf16 A and B, both
// K-major, N >> 3 and M >> 4.
DEVI uint32_t tc_idesc(uint32_t M, uint32_t N) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((N >> 3) << 17) | ((M >> 4) << 24);
}
DEVI void tc_mma(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc, uint32_t acc) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.u32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(acc)
      : "memory");
}
// arrives once on `bar` when every tensor-core operation this thread issued
// before it has completed
DEVI void tc_commit(uint64_t *bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                   saddr(bar))
               : "memory");
}
DEVI void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
DEVI void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }
DEVI void fence_proxy_async() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }
// 32 lanes x 16 columns of 32-bit words (this warp's lane quarter)
DEVI void tc_ld16(uint32_t taddr, float (&v)[16]) {
  uint32_t r[16];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}

DEVI void fence_mbar_init() { asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory"); }
DEVI uint64_t policy_evict_first() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}
// bulk async copy global -> this CTA's shared memory, completion counted in bytes on `bar`
DEVI void bulk_g2s(void *dst, const void *src, uint32_t bytes, uint64_t *bar, uint64_t pol) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1], %2, [%3], %4;" ::"r"(saddr(dst)),
      "l"(src), "r"(bytes), "r"(saddr(bar)), "l"(pol)
      : "memory");
}
DEVI uint32_t ld_acquire(const uint32_t *p) {
  uint32_t v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}
DEVI uint32_t ld_relaxed(const uint32_t *p) {
  uint32_t v;
  asm volatile("ld.relaxed.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}
DEVI void red_add(uint32_t *p, uint32_t v) {
  asm volatile("red.relaxed.gpu.global.add.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}
DEVI uint32_t atom_add_acq_rel(uint32_t *p, uint32_t v) {
  uint32_t old;
  asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v) : "memory");
  return old;
}
DEVI void fence_gpu() { asm volatile("fence.acq_rel.gpu;" ::: "memory"); }
// Release add: every write that happens before it (including other threads'
// writes ordered before it by a warp or block barrier) is visible to a thread
// that acquires the counter and sees the increment.
DEVI void red_release(uint32_t *p, uint32_t v) {
  asm volatile("red.release.gpu.global.add.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}
// SM cycle counter: cheap to read, used for every wait limit (the limits are
// budgeted at the maximum SM clock, so a limit is never shorter than stated)
DEVI uint64_t cycles() { return (uint64_t)clock64(); }
DEVI uint64_t gtimer() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}
DEVI uint32_t smid() {
  uint32_t s;
  asm volatile("mov.u32 %0, %%smid;" : "=r"(s));
  return s;
}
DEVI float bf_lo(uint32_t w) { return __uint_as_float(w << 16); }
DEVI float bf_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }
DEVI float bf1(uint16_t h) { return __uint_as_float((uint32_t)h << 16); }
DEVI uint16_t to_bf(float f) { return __bfloat16_as_ushort(__float2bfloat16_rn(f)); }
DEVI float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o; o >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, o);
  return v;
}
DEVI float warp_max(float v) {
#pragma unroll
  for (int o = 16; o; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xFFFFFFFFu, v, o));
  return v;
}

// ------------------------------------------------------- shared state ----
struct Smem {
  uint8_t *ring;
  uint64_t *full, *empty, *ifull, *iempty, *rdy, *done, *attbar, *xbar, *tbar, *dbar;
  uint64_t *bfull, *bempty;  // tensor-core B-operand slots written / read by the MMAs
  uint8_t *wring;            // stream plans: the compute warps' rings of 512-byte slots
  mk_instr *fifo;
  SlotMeta *meta;
  float *res, *opart, *ml, *sc, *rope, *normr, *rbuf, *xs;
  uint32_t *sat;
  int32_t *pos, *tok;
  uint64_t *dmask;     // attention re-deal: per chunk, the sequences it has work for
  uint32_t *dpre;      // and the prefix count of (chunk, sequence) pairs with work
  volatile int *misc;  // [0] bail, [1] bad input
  float *wsc;          // FP8 plans: the storer's copy of the current tile's row scales
};

static_assert(sizeof(Smem) <= kMiscDescBytes, "pointer table larger than its slot");

DEVI Smem make_smem(const KParams &P, uint8_t *base) {
  Smem S;
  S.ring = base;
  uint64_t *bars = reinterpret_cast<uint64_t *>(base + P.off_bars);
  const uint32_t E = P.ring_pages;
  S.full = bars;
  S.empty = bars + E;
  S.ifull = bars + 2 * E;
  S.iempty = S.ifull + kFifo;
  S.rdy = S.iempty + kFifo;
  S.done = S.rdy + kFifo;
  S.attbar = S.done + kFifo;
  S.xbar = S.attbar + 1;
  S.tbar = S.xbar + 1;  // tensor-core results of a tile ready
  S.dbar = S.tbar + 1;  // every tensor-core operation drained (kernel end)
  S.bfull = S.dbar + 1;
  S.bempty = S.bfull + kTcBufs;
  S.fifo = reinterpret_cast<mk_instr *>(base + P.off_fifo);
  S.meta = reinterpret_cast<SlotMeta *>(base + P.off_meta);
  S.res = reinterpret_cast<float *>(base + P.off_res);
  S.opart = reinterpret_cast<float *>(base + P.off_att);  // [2][warp][d]
  S.ml = S.opart + 2 * kComputeWarps * P.d;                  // [2][warp][m, l]
  S.sc = S.ml + 2 * kComputeWarps * 2;                       // [warp][att_lmax]
  S.sat = reinterpret_cast<uint32_t *>(base + P.off_sat);
  S.pos = reinterpret_cast<int32_t *>(base + P.off_pos);
  S.tok = S.pos + kMaxBatch;
  S.rope = reinterpret_cast<float *>(base + P.off_rope);
  S.normr = reinterpret_cast<float *>(base + P.off_normr);
  S.misc = reinterpret_cast<volatile int *>(base + P.off_misc);
  S.dmask = reinterpret_cast<uint64_t *>(base + P.off_deal);
  S.dpre = reinterpret_cast<uint32_t *>(S.dmask + kMaxDealChunks);
  S.rbuf = reinterpret_cast<float *>(base + P.off_rbuf);
  S.xs = reinterpret_cast<float *>(base + P.off_xs);
  S.wsc = reinterpret_cast<float *>(base + P.off_wsc);
  S.wring = base + P.off_wring;
  return S;
}

// where-codes for the latched error: role << 28 | instruction index
constexpr uint32_t kWhereLoader = 1u << 28, kWhereCompute = 2u << 28, kWhereStorer = 3u << 28,
                   kWherePoll = 4u << 28, kWhereDrain = 5u << 28;

DEVI void raise_error(const KParams &P, int code, uint32_t where, bool abort_all) {
  atomicCAS(P.ctrl + kCtlStatus, 0u, (uint32_t)code);
  atomicCAS(P.ctrl + kCtlWhere, 0u, where | 0x80000000u);
  if (abort_all) atomicExch(P.ctrl + kCtlAbort, 1u);
}

// One thread: stop if the block bails, the grid aborts, or the limit passed.
DEVI bool should_stop(const KParams &P, const Smem &S, uint64_t t0, uint32_t &n, uint32_t where) {
  if (S.misc[0]) return true;
  if ((++n & 7u) == 0) {
    if (ld_relaxed(P.ctrl + kCtlAbort)) {
      S.misc[0] = 1;
      return true;
    }
    if (cycles() - t0 > P.timeout_cycles) {
      raise_error(P, MK_ERR_TIMEOUT, where, true);
      S.misc[0] = 1;
      return true;
    }
  }
  return false;
}

// Single-thread bounded wait on an mbarrier phase.
DEVI bool thread_wait(const KParams &P, const Smem &S, uint64_t *bar, uint32_t parity,
                      uint32_t where) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = cycles();
  uint32_t n = 0;
  while (!mbar_try_wait(bar, parity))
    if (should_stop(P, S, t0, n, where)) return false;
  return true;
}

// Whole-warp bounded wait: every lane observes the phase itself (acquire);
// lane 0 decides on bailing and broadcasts it.
DEVI bool warp_wait(const KParams &P, const Smem &S, uint64_t *bar, uint32_t parity,
                    uint32_t where) {
  if (__all_sync(0xFFFFFFFFu, mbar_try_wait(bar, parity))) return true;
  const uint64_t t0 = cycles();
  uint32_t n = 0;
  while (true) {
    if (__all_sync(0xFFFFFFFFu, mbar_try_wait(bar, parity))) return true;
    int stop = 0;
    if ((threadIdx.x & 31) == 0) stop = should_stop(P, S, t0, n, where);
    if (__shfl_sync(0xFFFFFFFFu, stop, 0)) return false;
  }
}

// ----------------------------------------------------- attention range ----
// Chunk c covers positions [c * attn_chunk, (c + 1) * attn_chunk) of 0..pos:
// the chunks past p_b are empty (their instructions only take part in the
// arrival), so a short sequence of a ragged batch costs few chunks.
DEVI void attn_range(const KParams &P, int pos, int c, int &p0, int &p1) {
  p0 = c * P.attn_chunk;
  p1 = min(p0 + P.attn_chunk, pos + 1);
  if (p1 < p0) p1 = p0;
}

DEVI size_t kv_row(const KParams &P, int l, int b, int g, int p) {
  return ((((size_t)l * P.B + b) * P.nkv + g) * P.max_ctx + p) * P.d;
}

// -------------------------------------------------------------- compute ----
// Wait for the instruction's input counter (one thread).  `sat` caches the
// last satisfied absolute target per waited counter for this launch.
DEVI bool poll_counter(const KParams &P, const Smem &S, const mk_instr &in, uint32_t epoch,
                       uint32_t idx) {
  if (P.mode == kModeRange || in.wait_ctr == MK_NO_COUNTER) return true;
  const uint32_t c = in.wait_ctr;
  // counters are never reset: this step's target sits on top of the
  // epoch * (signals per step) the counter received in earlier steps
  const uint32_t target = epoch * __ldg(P.ctr_inc + c) + in.wait_tgt;
  const bool cacheable = c < (uint32_t)P.n_wait;
  if (cacheable && S.sat[c] != 0 && (int32_t)((S.sat[c] - 1u) - target) >= 0) return true;
  const uint32_t *p = P.ctr + (size_t)c * kCtrStride;
  bool ok = (int32_t)(ld_acquire(p) - target) >= 0;
  if (!ok) {
    const uint64_t t0 = cycles();
    uint32_t n = 0;
    while (true) {
      __nanosleep(20);
      if ((int32_t)(ld_acquire(p) - target) >= 0) {
        ok = true;
        break;
      }
      if (should_stop(P, S, t0, n, kWherePoll | idx)) return false;
    }
  }
  if (cacheable) S.sat[c] = target + 1u;
  return true;
}

struct XCache {
  float v[kMaxChunks][8];
};

DEVI const uint16_t *gain_of(const KParams &P, int op, int layer) {
  if (op == MK_OP_QKV) return P.norms + (size_t)(2 * layer) * P.H;
  if (op == MK_OP_GATEUP) return P.norms + (size_t)(2 * layer + 1) * P.H;
  if (op == MK_OP_LMHEAD) return P.norms + (size_t)(2 * P.L) * P.H;
  return nullptr;
}

// 8 consecutive input values of sequence b at column col
DEVI void load8(const KParams &P, const Smem &S, int op, int emb, int b, int col, float (&v)[8]) {
  if (emb) {
    const uint4 w = __ldg(reinterpret_cast<const uint4 *>(P.embed + (size_t)S.tok[b] * P.H + col));
    v[0] = bf_lo(w.x); v[1] = bf_hi(w.x); v[2] = bf_lo(w.y); v[3] = bf_hi(w.y);
    v[4] = bf_lo(w.z); v[5] = bf_hi(w.z); v[6] = bf_lo(w.w); v[7] = bf_hi(w.w);
    return;
  }
  const float *src;
  if (op == MK_OP_OPROJ) src = P.attn + (size_t)b * P.nq * P.d;
  else if (op == MK_OP_DOWN) src = P.h + (size_t)b * P.F;
  else src = P.x + (size_t)b * P.H;
  const float4 a = __ldcg(reinterpret_cast<const float4 *>(src + col));
  const float4 c = __ldcg(reinterpret_cast<const float4 *>(src + col + 4));
  v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w; v[4] = c.x; v[5] = c.y; v[6] = c.z; v[7] = c.w;
}

DEVI void load_gain8(const uint16_t *g, int col, float (&v)[8]) {
  const uint4 w = __ldg(reinterpret_cast<const uint4 *>(g + col));
  v[0] = bf_lo(w.x); v[1] = bf_hi(w.x); v[2] = bf_lo(w.y); v[3] = bf_hi(w.y);
  v[4] = bf_lo(w.z); v[5] = bf_hi(w.z); v[6] = bf_lo(w.w); v[7] = bf_hi(w.w);
}

// Batch 1: the warp's input slice, normalised and scaled by the gains, kept
// in registers for as long as consecutive instructions share the input.
// Split in two so the gains (constants) are loaded before the dependency
// wait and only the activations are fetched after it, in one round trip.
DEVI uint32_t input_key(const mk_instr &in) {
  return ((uint32_t)in.op << 24) | ((uint32_t)(in.flags & 1) << 23) | in.layer;
}

// Barrier of the compute warps on an mbarrier (bounded).
DEVI bool compute_sync(const KParams &P, const Smem &S, uint64_t *bar, uint32_t &uses, int lane) {
  __syncwarp();
  if (lane == 0) mbar_arrive(bar);
  const bool ok = warp_wait(P, S, bar, uses & 1u, kWhereCompute);
  ++uses;
  return ok;
}

// Wait for FIFO entry fs (idempotent: may be called again for the same
// entry).  The entry stays in shared memory, read in place, until the
// storer releases the slot.
DEVI bool next_entry(const KParams &P, const Smem &S, uint32_t fs) {
  const uint32_t f = fs % kFifo, k = fs / kFifo;
  return warp_wait(P, S, &S.ifull[f], k & 1u, kWhereCompute);
}

// Dependency wait of entry fs: compute warp 0 polls the counter, the others
// wait on the slot's ready barrier.
DEVI bool ready_entry(const KParams &P, const Smem &S, uint32_t fs, const mk_instr &in,
                      const SlotMeta &meta, uint32_t epoch, int cw, int lane) {
  const uint32_t f = fs % kFifo, k = fs / kFifo;
  if (cw == 0) {
    int ok = 1;
    if (lane == 0) {
      ok = poll_counter(P, S, in, epoch, meta.idx);
      if (ok) {
        if (P.flags & MK_FLAG_TRACE) S.meta[f].t_ready = gtimer();
        mbar_arrive(&S.rdy[f]);
      }
    }
    if (!__shfl_sync(0xFFFFFFFFu, ok, 0)) return false;
  }
  return warp_wait(P, S, &S.rdy[f], k & 1u, kWhereCompute | meta.idx);
}

DEVI void finish_entry(const KParams &P, const Smem &S, uint32_t fs, int cw, int lane) {
  __syncwarp();
  if (lane == 0) {
    if (cw == 0 && (P.flags & MK_FLAG_TRACE)) S.meta[fs % kFifo].t_cdone = gtimer();
    mbar_arrive(&S.done[fs % kFifo]);
  }
}

// --------------------------------------------------------------- storer ----
// Q8: FP8 weights; a tile row's sum is multiplied by the row's scale (the
// storer copied the tile's scales into S.wsc while the compute warps ran).
template <bool Q8 = false>
DEVI void storer_epilogue(const KParams &P, const Smem &S, const mk_instr &in,
                          const SlotMeta &meta, const float *res, int lane, uint32_t epoch) {
  const int B = P.B, d = P.d;
  const OpGeom &G = P.geom[in.op];
  auto val = [&](uint32_t r, int b) {
    float v = 0.f;
    for (uint32_t s = 0; s < G.NS; ++s) v += res[(r * G.NS + s) * B + b];
    if (Q8) v *= S.wsc[r];
    return v;
  };
  uint32_t *ctr = P.ctr;
  // batch > 1 projections finish (and signal) on the compute warps
  const bool compute_owned = in.op == MK_OP_ATTN || P.tc;
  if (!compute_owned) switch (in.op) {
    case MK_OP_QKV: {
      // rows come in pairs: one RoPE rotation pair (natural dims i and
      // i + d/2) of a q head or of k, or two consecutive v dims
      const int GR = (P.qpg + 2) * d, half = d / 2;
      const int npairs = (int)in.nrows / 2;
      for (int u = lane; u < npairs * B; u += 32) {
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
      // residual rows were prefetched into rbuf by this lane (same u mapping)
      for (int u = lane; u < (int)in.nrows * B; u += 32) {
        const int r = u % in.nrows, b = u / in.nrows;
        P.x[(size_t)b * P.H + in.row0 + r] = S.rbuf[u] + val(r, b);
      }
      break;
    }
    case MK_OP_GATEUP: {
      for (int u = lane; u < (int)in.nrows * B; u += 32) {
        const int j = u % in.nrows, b = u / in.nrows;
        const float gt = val(j, b), up = val(in.nrows + j, b);
        P.h[(size_t)b * P.F + in.row0 + j] = gt / (1.f + __expf(-gt)) * up;
      }
      break;
    }
    case MK_OP_LMHEAD: {
      for (int u = lane; u < (int)in.nrows * B; u += 32) {
        const int r = u % in.nrows, b = u / in.nrows;
        P.logits[(size_t)b * P.V + in.row0 + r] = val(r, b);
      }
      break;
    }
    case MK_OP_ATTN:
      break;  // the compute warps wrote the chunk partial to global memory
  }
  // the warp barrier orders every lane's output writes before lane 0's
  // release (the compute warps' chunk partials were ordered before this
  // warp by the slot's done barrier)
  // (attention chunks signal and merge from the compute warps)
  __syncwarp();
  if (!compute_owned && lane == 0) red_release(ctr + (size_t)in.sig_ctr * kCtrStride, 1u);
  if (lane == 0) {
    red_add(P.exec + meta.idx, 1u);
    if (P.flags & MK_FLAG_TRACE) {
      unsigned long long *tr = P.trace + (size_t)meta.idx * kTraceWords;
      tr[0] = ((unsigned long long)smid() << 32) | blockIdx.x;
      tr[1] = meta.t_claim;
      tr[2] = meta.t_ready;
      tr[3] = gtimer();
      tr[4] = meta.t_issued;
      tr[5] = meta.t_cdone;
      tr[6] = meta.t_sstart;
      tr[7] = meta.t_input;
      tr[8] = meta.t_page0;
      tr[9] = meta.t_pagel;
    }
  }
}

// Residual rows of an O/down instruction, fetched while the compute warps
// work on it (its input counter is satisfied once the slot is ready).
DEVI void prefetch_residual(const KParams &P, const Smem &S, const mk_instr &in, int lane) {
  if (in.op != MK_OP_OPROJ && in.op != MK_OP_DOWN) return;
  const int n = (int)in.nrows * P.B;
#pragma unroll 4
  for (int u = lane; u < n; u += 32) {
    const int r = u % in.nrows, b = u / in.nrows, row = in.row0 + r;
    S.rbuf[u] = (in.op == MK_OP_OPROJ && (in.flags & 1))
                    ? bf1(P.embed[(size_t)S.tok[b] * P.H + row])
                    : __ldcg(P.x + (size_t)b * P.H + row);
  }
}

}  // namespace mk
