// mk_internal.h -- definitions shared by the planner, the host runtime and the
// megakernel of libmk.so.  Nothing here is part of the public ABI (mk.h).
#pragma once
#include <stdint.h>

#include "mk.h"

namespace mk {

// Block shape: warp 0 = loader, warp 1 = storer, warps 2.. = compute.
// Roles after « 5 · La spécialisation des warps », §5.4 (loader, compute,
// storer; the scheduler role is the loader's queue claim).
constexpr int kComputeWarps = 14;  // 16 warps per block: 4 per SM sub-partition, 128 registers each
constexpr int kThreads = 32 * (2 + kComputeWarps);
constexpr int kFifo = 8;        // instructions a block may hold ahead of compute
constexpr int kMaxBatch = 48;   // 1..16, or 32 / 48 (tensor-core readback in blocks of 16)
constexpr int kMaxQpg = 8;      // q heads per KV group
constexpr int kMaxItems = 256;  // work items (row x slice) per GEMV instruction
constexpr int kMaxItemsB = 256; // work items x batch per GEMV instruction
constexpr int kMaxChunks = 4;   // 256-column chunks per item: the input slice a lane keeps in
                                // registers (8 per chunk); 4 keeps the GEMV loop free of spills
constexpr int kTcBufs = 4;     // ring slots of the tensor-core B operand (one page's columns each)
constexpr int kCtrStride = 32;  // u32 words between counters (128 B apart)
constexpr int kMaxRing = 32;
constexpr int kMaxDealChunks = 256;  // attention chunks per (sequence, group) the re-deal tabulates
// stream plans: each compute warp's ring of 512-byte slots is filled by
// per-lane async copies in commit groups of kSG slots
constexpr int kSG = 4;
constexpr int kMaxWarpRing = 32;  // slots per warp ring (at most 8 commit groups in flight)
// block flags (bail, bad input) at the start of the misc area, then the
// table of the block's shared-memory pointers
constexpr int kMiscDescOffset = 64, kMiscDescBytes = 256;

// control words (u32 index into the ctrl block)
constexpr int kCtlStatus = 0, kCtlWhere = 1, kCtlAbort = 2, kCtlEpoch = 3;
constexpr int kCtlExit = 32, kCtlQueue = 64, kCtlWords = 96;

// run modes
constexpr int kModeDynamic = 0, kModeStatic = 1, kModeRange = 2, kModeHybrid = 3;

// GEMV geometry of one op: K input columns split into NS slices of SW
// columns; an item = one weight row restricted to one slice (2*SW bytes);
// ipp items are packed per shared-memory page; nch = SW/256 16-byte chunks
// per lane.
struct OpGeom {
  uint32_t K, NS, SW, item_bytes, ipp, nch;
  // batch > 1 (tensor-core) plans: blocks of MR weight rows stored as kp
  // pages of MR rows x kc columns in the MMA's core-matrix order; a block is
  // split along K into S slices of whole pages (slice s: pages
  // [s kp / S, (s + 1) kp / S))
  uint32_t MR, S, kc, kp;
};

struct KParams {
  const mk_instr *instr;
  uint32_t n_instr;
  const uint32_t *list_off, *list_idx;
  uint32_t *aq;                // hybrid: per-layer attention queue (claims, epoch relative)
  const uint32_t *att_first;   // hybrid: per layer, first instruction of its attention phase
  uint32_t att_count;          // attention instructions per layer
  uint32_t *ctr, *ctrl, *exec;
  const uint32_t *ctr_inc;  // signals per step of every counter
  unsigned long long *trace;
  const uint8_t *arena;
  const uint16_t *embed;   // plain [V][H]
  const uint16_t *norms;   // [L][2][H] then final [H]
  uint16_t *kc, *vc;       // [L][B][nkv][max_ctx][d]
  const int32_t *tokens, *positions;
  float *logits;
  float *x, *q, *attn, *h, *part;
  const float *rope_cos, *rope_sin;  // [max_ctx][d/2]
  OpGeom geom[8];
  int32_t L, H, nq, nkv, d, F, V, B, max_ctx, qpg;
  int32_t nchunk, attn_chunk, att_lmax;
  int32_t tc, tc_nb;  // tensor-core projections (batch > 1); MMA N = 2 x batch rounded up to 16
  int32_t stream;     // batch 1: compute warps stream their own weights (per-warp rings)
  int32_t att_grp;
  uint32_t tmem_cols;  // tensor-core plans: tensor-memory columns of the accumulator    // attention warps serve all query heads of the group (attn_chunk_grp)
  uint32_t wnb;       // stream plans: slots (512 B) in each compute warp's ring
  float *gpart;       // partial sums of split projections [block][slice][MR][B]
  float eps, attn_scale;
  int32_t n_wait, mode;
  uint32_t range_first, range_count, n_blocks, flags;
  uint64_t timeout_cycles;  // wait limit in SM cycles (at the maximum SM clock)
  uint32_t lookahead;  // FIFO entries the loader may publish ahead of its stream
  uint32_t l2_window;  // bytes of published pages prefetched into L2 ahead of the ring
  uint32_t loader_idle_ns;  // back-off of the loader thread when it can make no progress
  // dynamic shared-memory layout (byte offsets)
  uint32_t ring_pages, page_bytes;
  uint32_t off_bars, off_fifo, off_meta, off_res, res_floats, off_att, off_sat, off_pos,
      off_rope, off_normr, off_misc, off_rbuf, off_xs, off_wring, off_deal, smem_total;
  int32_t fp8;       // batch 1: FP8 E4M3 weight codes with one scale per row (MK_FLAG_FP8_WEIGHTS)
  uint32_t off_wsc;  // FP8 plans: the storer's row-scale buffer in shared memory
};

// per FIFO slot metadata written by the loader
struct SlotMeta {
  uint32_t idx, seq0, npages, pad;
  // trace timestamps (%globaltimer, MK_FLAG_TRACE only): published by the
  // loader, last page issued, input ready, compute done, storer start
  unsigned long long t_claim, t_issued, t_ready, t_cdone, t_sstart, t_input, t_page0, t_pagel;
};
constexpr int kTraceWords = 10;  // u64 per instruction in the trace buffer

#ifdef __CUDACC__
cudaError_t set_megakernel_smem(uint32_t bytes);
cudaError_t launch_row_scale(uint8_t *dst, const uint8_t *src, const int32_t *map,
                             const uint64_t *scaletab, uint32_t nrows, uint32_t K,
                             cudaStream_t stream);
cudaError_t launch_retile_q8(uint8_t *dst, const uint8_t *src, const int32_t *map,
                             const uint64_t *rowtab, const uint64_t *scaletab, uint32_t nrows,
                             const OpGeom &g, uint32_t page, cudaStream_t stream);
cudaError_t launch_megakernel(const KParams &P, uint32_t grid, bool cooperative,
                              cudaStream_t stream);
cudaError_t launch_epoch_advance(uint32_t *ctrl, cudaStream_t stream);
cudaError_t launch_retile_tc(uint8_t *dst, const uint8_t *src, const int32_t *map,
                             uint32_t nrows, const OpGeom &g, uint32_t page, cudaStream_t stream);
cudaError_t launch_retile(uint8_t *dst, const uint8_t *src, const int32_t *map,
                          const uint64_t *rowtab, uint32_t nrows, const OpGeom &g, uint32_t page,
                          cudaStream_t stream);
cudaError_t launch_retile_stream(uint8_t *dst, const uint8_t *src, const int32_t *map,
                                 const uint64_t *rowtab, uint32_t nrows, const OpGeom &g,
                                 cudaStream_t stream);
cudaError_t set_stream_smem(uint32_t bytes);
cudaError_t launch_megakernel_stream(const KParams &P, uint32_t grid, bool cooperative,
                                     cudaStream_t stream);
#endif

}  // namespace mk
