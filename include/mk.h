/*
 * mk.h -- C ABI of the persistent decode megakernel library (libmk.so).
 *
 * One call of mk_decode_step() enqueues ONE kernel launch that runs a whole
 * Llama-style decoder forward pass for a small batch of sequences: the
 * megakernel of « 2 · Définition et généalogie », §2.1 (one launch,
 * persistent, fine-grained dependencies in global memory, internal
 * heterogeneity by dispatch).  The host builds the instruction list (§2.5,
 * the anatomy figure: "CPU : construit la liste d'instructions"); one block
 * per SM interprets it (§2.6, "2. Le dispatch d'instructions"), streaming
 * weights through a paged shared-memory ring (§2.6, "4. L'allocateur de
 * mémoire partagée") with warp-specialised loader / compute / storer roles
 * (« 5 · La spécialisation des warps », §5.2 and §5.4), and kernel boundaries
 * are replaced by dependency counters (§2.6, "3. Les compteurs de
 * dépendance") and a global work queue (§2.4; §2.6, "5. L'ordonnancement").
 *
 * Conventions for every call:
 *  - Returns MK_OK (0) or a negative MK_ERR_* code; mk_error_string() names it.
 *    No C++ exception crosses this boundary.
 *  - "device pointer" = CUDA global memory of the current device; "host
 *    pointer" = ordinary or pinned host memory.  `stream` is a cudaStream_t
 *    passed as void* (NULL = the legacy default stream).
 *  - bf16 tensors are passed as raw 16-bit patterns (uint16_t storage).
 *  - The library allocates only inside an opaque plan (re-tiled weights,
 *    instruction/counter tables, activations, staging); the caller owns every
 *    buffer it passes in and keeps ownership.
 *  - A call that fails host-side validation launches nothing.
 */
#ifndef MK_H
#define MK_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#if defined(__GNUC__)
#define MK_API __attribute__((visibility("default")))
#else
#define MK_API
#endif

/* ---- return codes ------------------------------------------------------- */
#define MK_OK 0
#define MK_ERR_CONFIG -1  /* configuration the library cannot plan */
#define MK_ERR_ARG -2     /* NULL or inconsistent argument */
#define MK_ERR_DEVICE -3  /* no usable sm_103 device, or device query failed */
#define MK_ERR_NOMEM -4   /* device or host allocation failed */
#define MK_ERR_STATE -5   /* call out of order (e.g. step before weights) */
#define MK_ERR_TIMEOUT -6 /* a device-side wait exceeded wait_timeout_us */
#define MK_ERR_BOUNDS -7  /* a token or position was out of range on device */
#define MK_ERR_LAUNCH -8  /* kernel launch rejected */
#define MK_ERR_CUDA -9    /* other CUDA runtime error */

/* ---- opcodes of the instruction table (field `op`) ---------------------- */
#define MK_OP_END 0     /* end of work (device-internal, never in a table) */
#define MK_OP_QKV 1     /* RMSNorm + fused q/k/v GEMV + RoPE + KV append */
#define MK_OP_ATTN 2    /* GQA decode attention over one KV chunk (+ group merge) */
#define MK_OP_OPROJ 3   /* x += Wo . attn */
#define MK_OP_GATEUP 4  /* RMSNorm + gate/up GEMV + SiLU(gate) * up */
#define MK_OP_DOWN 5    /* x += Wd . h */
#define MK_OP_LMHEAD 6  /* final RMSNorm + LM-head GEMV -> logits */

#define MK_NO_COUNTER 0xFFFFFFFFu

/* ---- flags (mk_config.flags) --------------------------------------------- */
#define MK_FLAG_TRACE 0x1u      /* record per-instruction timestamps (mk_read_trace) */
#define MK_FLAG_HOST_ONLY 0x2u  /* build the tables only; no CUDA call at all */
#define MK_FLAG_FAULT_WAIT 0x4u /* TEST ONLY: one wait target is made unreachable */
#define MK_FLAG_STREAM_B1 0x8u  /* batch 1: every compute warp streams its own weights through
                                   a private ring of per-lane async copies, instead of the
                                   block's shared page ring fed by the loader warp's bulk
                                   copies (the default); an alternative kept for comparison */
#define MK_FLAG_FP8_WEIGHTS 0x10u /* batch 1, shared page ring: every projection and the LM
                                     head streamed as FP8 E4M3 codes with one float scale per
                                     output row (scale = row amax / 448, code = E4M3 of w /
                                     scale, round to nearest even, saturating), quantised by
                                     mk_load_weights from the bf16 weights; the embedding
                                     lookup, the norms and the KV cache stay bf16.  The pages'
                                     "lower precision" lever (« Résumé exécutif », "Les six
                                     leviers"); results differ from bf16 by the weights'
                                     quantisation.  MK_ERR_CONFIG for batch > 1 or with
                                     MK_FLAG_STREAM_B1 */

#define MK_SCHED_DYNAMIC 0 /* global work queue, one atomic claim per instruction */
#define MK_SCHED_STATIC 1  /* per-SM lists, round-robin over the queue order */
#define MK_SCHED_HYBRID 2  /* per-SM lists for the projections; each layer's attention
                              chunks claimed from that layer's own queue, one claim at
                              a time as a block's instruction FIFO drains (the pages'
                              hybrid of static and dynamic scheduling, « 2 · Définition
                              et généalogie », §2.6 "5. L'ordonnancement"); not with
                              MK_FLAG_STREAM_B1 */

/* Model shape and plan options.  A plan is built for one batch size
   (« Résumé exécutif », "Où en est-on en 2026": a megakernel is rebuilt per
   batch size). */
typedef struct mk_config {
  int32_t n_layers, hidden, n_q_heads, n_kv_heads, head_dim, ffn_dim, vocab;
  float rms_eps, rope_theta;
  int32_t tie_embeddings;  /* 1: the LM head is the embedding matrix */
  int32_t batch;           /* sequences per step: 1..16, or 32 or 48 (larger-batch mode:
                              tensor cores, 16 KB pages unless page_bytes says otherwise) */
  int32_t max_ctx;         /* KV capacity per sequence (positions), multiple of 16 */
  int32_t sched_mode;      /* MK_SCHED_DYNAMIC, MK_SCHED_STATIC or MK_SCHED_HYBRID */
  uint32_t flags;          /* MK_FLAG_* */
  int32_t wait_timeout_us; /* device-side wait limit; 0 -> 1,000,000 */
  int32_t num_sms;         /* 0 -> query the device; >0 overrides (host-only planning) */
  int32_t smem_bytes;      /* 0 -> device opt-in maximum per block */
  int32_t page_bytes;      /* shared-memory page size; 0 -> 32768 */
  int32_t attn_chunk;      /* max KV positions per attention instruction; 0 -> auto */
  int32_t l2_prefetch_kb;  /* per block: KB of published pages prefetched into L2 ahead of
                              the shared-memory ring; <= 0 -> none (the default: on the
                              batch-1 workloads the extra L2 traffic costs more than it hides) */
} mk_config;

/* One instruction: a fixed 64-byte little-endian record.
   Output rows: QKV -> rows of the fused q/k/v output, grouped per KV head g
   (the q heads g*qpg..g*qpg+qpg-1, then k head g, then v head g, d rows
   each); GATEUP -> FFN activations h; OPROJ, DOWN -> residual rows; LMHEAD ->
   vocabulary rows.  An ATTN instruction covers chunk `chunk` of `nchunk` of
   the KV positions 0..pos_b of sequence b, group g; it adds 1 to its group's
   arrival counter `sig_ctr`, and the chunk that completes the group (the
   nchunk-th arrival of the step) merges the group and adds 1 to `sig2_ctr`.
   Waits are per step: the instruction may start once counter `wait_ctr` has
   received `wait_tgt` signals in the current step (targets are epoch
   relative, counters are never reset between steps). */
typedef struct mk_instr {
  uint8_t op;          /*  0 MK_OP_* */
  uint8_t flags;       /*  1 bit 0: input/residual is the embedding row (layer 0) */
  uint16_t layer;      /*  2 */
  uint16_t b;          /*  4 sequence (ATTN) */
  uint16_t g;          /*  6 KV group (QKV, ATTN) */
  uint32_t wait_ctr;   /*  8 counter id or MK_NO_COUNTER */
  uint32_t wait_tgt;   /* 12 signals required in this step */
  uint32_t sig_ctr;    /* 16 counter signalled (+1) on completion */
  uint32_t sig2_ctr;   /* 20 ATTN: group-merge counter, else MK_NO_COUNTER */
  uint32_t sig2_after; /* 24 ATTN: arrivals per step that complete the group */
  uint32_t row0;       /* 28 first output row */
  uint32_t nrows;      /* 32 output rows */
  uint32_t chunk;      /* 36 ATTN chunk index */
  uint32_t nchunk;     /* 40 ATTN chunks per (sequence, group) */
  uint32_t npages;     /* 44 weight pages streamed (GEMV ops; ATTN: 0, set at run time) */
  uint64_t wofs;       /* 48 byte offset of the tile's first page in the weight arena */
  uint32_t phase;      /* 56 index of the op phase (one launch in the multi-kernel path) */
  uint32_t reserved;   /* 60 zero */
} mk_instr;

/* A contiguous run of the queue holding one op of one layer. */
typedef struct mk_phase {
  uint32_t first, count, op, layer;
} mk_phase;

typedef struct mk_plan_info_s {
  uint32_t n_instr, n_counters, n_wait_counters, n_phases;
  uint32_t n_blocks;        /* persistent grid = SMs used, one block each */
  uint32_t threads;         /* per block: 1 loader warp + 1 storer warp + compute warps */
  uint32_t ring_pages;      /* pages in the shared-memory ring */
  uint32_t page_bytes;
  uint32_t fifo_depth;      /* instructions a block may hold ahead of its compute warps */
  uint32_t smem_bytes;      /* dynamic shared memory per block */
  uint32_t attn_nchunk;     /* attention chunks per (sequence, group) */
  uint32_t attn_chunk;      /* max positions per chunk */
  uint64_t arena_bytes;     /* re-tiled weights held by the plan */
  uint64_t weight_bytes;    /* algorithmic weight bytes streamed per step (FP8 plans: codes
                               and row scales) */
  uint32_t warp_ring_slots; /* MK_FLAG_STREAM_B1 plans: 512-byte slots in each compute
                               warp's ring (0: the plan uses the shared page ring) */
  uint32_t kernel;          /* 0 shared page ring (batch 1, the default), 1 tensor cores
                               (batch > 1), 2 per-warp streams (batch 1, MK_FLAG_STREAM_B1),
                               3 shared page ring with FP8 weights (MK_FLAG_FP8_WEIGHTS) */
} mk_plan_info_t;

/* Weights in PyTorch layout ([out, in] row-major, bf16 bit patterns), as host
   or device pointers.  mk_load_weights copies and re-tiles them into
   plan-owned device memory; the caller keeps its buffers. */
typedef struct mk_layer_weights {
  const void *attn_norm; /* [H] */
  const void *wq;        /* [nq*d, H] */
  const void *wk;        /* [nkv*d, H] */
  const void *wv;        /* [nkv*d, H] */
  const void *wo;        /* [H, nq*d] */
  const void *mlp_norm;  /* [H] */
  const void *w_gate;    /* [F, H] */
  const void *w_up;      /* [F, H] */
  const void *w_down;    /* [H, F] */
} mk_layer_weights;

typedef struct mk_weights {
  const void *embed;               /* [V, H] */
  const void *final_norm;          /* [H] */
  const void *lm_head;             /* [V, H]; NULL when tie_embeddings */
  const mk_layer_weights *layers;  /* host array of n_layers entries */
} mk_weights;

/* Caller-owned KV cache, device pointers, each [L][B][nkv][max_ctx][d] bf16.
   Keys are stored after RoPE. */
typedef struct mk_kv_cache {
  void *k;
  void *v;
} mk_kv_cache;

/* Device pointers to the plan's activation buffers (fp32), for per-op tests. */
typedef struct mk_debug_buffers_s {
  float *x;    /* [B][H] residual stream */
  float *q;    /* [B][nq][d] rotated queries */
  float *attn; /* [B][nq*d] attention output */
  float *h;    /* [B][F] SiLU(gate)*up */
} mk_debug_buffers_t;

typedef struct mk_plan_s *mk_plan_t;

/* Text for a return code.  Never NULL; static storage. */
MK_API const char *mk_error_string(int code);

/* Build the instruction, counter and phase tables for `cfg` on the host and,
   unless MK_FLAG_HOST_ONLY, allocate the plan's device state on the current
   device and upload the tables and the RoPE table.  Errors: MK_ERR_ARG (NULL),
   MK_ERR_CONFIG (shape not plannable: hidden/ffn not multiples of 256,
   n_q_heads not a multiple of n_kv_heads or more than 8 q heads per group,
   head_dim not 64 or 128, batch not in 1..16 or 32 or 48, max_ctx not a positive
   multiple of 16, shared memory too small), MK_ERR_DEVICE (not an sm_103
   device), MK_ERR_NOMEM.  On success *out owns everything; free it with
   mk_destroy. */
MK_API int mk_plan(const mk_config *cfg, mk_plan_t *out);

/* Plan geometry (see mk_plan_info_t). */
MK_API int mk_plan_info(mk_plan_t plan, mk_plan_info_t *info);

/* Host copies owned by the plan: the instruction table in queue order and
   the number of signals each counter receives per step (for replay checks).
   Pointers stay valid until mk_destroy. */
MK_API int mk_plan_tables(mk_plan_t plan, const mk_instr **instr, size_t *n_instr,
                          const uint32_t **counter_inc, size_t *n_counters);

/* Phase table (queue order) and static per-SM lists: list s holds
   list_idx[list_off[s] .. list_off[s+1]); n_lists = n_blocks.  In
   MK_SCHED_HYBRID plans every list holds, in place of layer l's attention
   instructions, one entry MK_LIST_ATTN | l: there the block claims chunks
   from layer l's attention queue until it is empty. */
#define MK_LIST_ATTN 0x80000000u
MK_API int mk_plan_phases(mk_plan_t plan, const mk_phase **phases, size_t *n_phases);
MK_API int mk_plan_lists(mk_plan_t plan, const uint32_t **list_off, const uint32_t **list_idx,
                         size_t *n_lists);

/* Copy and re-tile the weights (host or device pointers, see mk_weights)
   into plan-owned memory: q/k rows are paired for RoPE, gate/up rows are
   interleaved per tile, every tile is laid out as whole shared-memory pages.
   The pages' statement of the problem (« Résumé exécutif », "Le problème")
   is batch-1 decode bound by streaming every bf16 weight byte once per
   step; this call lays the weights out in the order the loader streams them
   (« 2 · Définition et généalogie », §2.6, "4. L'allocateur de mémoire
   partagée": pages of a shared-memory ring).
   Synchronises `stream` before returning.  Errors: MK_ERR_ARG, MK_ERR_STATE
   (host-only plan), MK_ERR_NOMEM, MK_ERR_CUDA. */
MK_API int mk_load_weights(mk_plan_t plan, const mk_weights *w, void *stream);

/* One decode step, asynchronous on `stream`; enqueues exactly one kernel
   launch (grid = n_blocks, one resident block per SM, cooperative launch so
   the driver refuses a grid that cannot be co-resident): the whole forward
   pass in one persistent launch (« 2 · Définition et généalogie », §2.1 and
   §2.4, persistent threads; §2.6 "1. La persistance").
     tokens    device int32 [B]     token of each sequence
     positions device int32 [B]     position p_b; the step writes K/V at p_b and
                                    attends to positions 0..p_b
     kv        caller-owned cache (device pointers)
     logits    device fp32 [B][V]   written
   Tokens outside [0,V) or positions outside [0,max_ctx) are detected on the
   device: nothing is computed and mk_status reports MK_ERR_BOUNDS.
   Host-side errors: MK_ERR_ARG, MK_ERR_STATE (weights not loaded),
   MK_ERR_LAUNCH. */
MK_API int mk_decode_step(mk_plan_t plan, const int32_t *tokens, const int32_t *positions,
                          const mk_kv_cache *kv, float *logits, void *stream);

/* The same step with HOST buffers: copies tokens and positions to the device,
   launches, copies the logits back and synchronises `stream`.  tokens and
   positions are host int32 [B], logits host fp32 [B][V] (pinned memory makes
   the copies asynchronous).  Returns host-side errors as mk_decode_step does;
   errors found on the device are reported by mk_status. */
MK_API int mk_decode_step_host(mk_plan_t plan, const int32_t *tokens, const int32_t *positions,
                               const mk_kv_cache *kv, float *logits, void *stream);

/* Baseline: the same step as one kernel launch per op phase (5 per layer + 1)
   with the same device functions and no cross-phase prefetch; with
   use_graph != 0 the launches are captured once into a CUDA graph (per set
   of argument pointers) and replayed.  Same arguments and errors as
   mk_decode_step. */
MK_API int mk_multikernel_step(mk_plan_t plan, const int32_t *tokens, const int32_t *positions,
                               const mk_kv_cache *kv, float *logits, int use_graph,
                               void *stream);

/* Run phase `phase` of the table alone as one launch (per-op tests).  It
   signals its counters but does not advance the step epoch; call mk_reset
   before a full step afterwards. */
MK_API int mk_run_phase(mk_plan_t plan, int phase, const int32_t *tokens,
                        const int32_t *positions, const mk_kv_cache *kv, float *logits,
                        void *stream);

/* Synchronise `stream` and return the first device error latched since the
   last call (MK_ERR_TIMEOUT, MK_ERR_BOUNDS) or MK_OK.  After a device error
   the counters, queue, epoch and execution counts are reset so the plan can
   run again.  The pages note that counter waits make progress only while
   every block is resident (« 2 · Définition et généalogie », §2.6 "1. La
   persistance" and the chapter's questions on deadlock); every wait here is
   bounded and reports MK_ERR_TIMEOUT instead of hanging. */
MK_API int mk_status(mk_plan_t plan, void *stream);

/* Synchronise the device and copy out, for bit-exact checks: counters
   (n_counters u32), the work-queue counter, per-instruction execution counts
   (n_instr u32) and the step epoch.  Any pointer may be NULL.  The counters
   are the dependency counters of « 2 · Définition et généalogie », §2.6 "3.
   Les compteurs de dépendance" (a producer adds 1 after its data is visible,
   a consumer waits for a target); the queue is the global work queue of §2.6
   "5. L'ordonnancement". */
MK_API int mk_read_counters(mk_plan_t plan, uint32_t *counters, uint32_t *queue, uint32_t *exec,
                            uint32_t *epoch);

/* With MK_FLAG_TRACE: n_instr records of 10 u64 {sm id << 32 | block,
   t_published, t_ready, t_done, t_pages_issued, t_compute_done,
   t_storer_start, s1, s2, s3} (%globaltimer ns) of the last step.  The
   stage stamps s1..s3: a batch-1 GEMV, input in registers, first page
   present, last page present; a tensor-core tile, MMA loop entered, first
   page present, last page's B operand present; an attention chunk with work,
   query and current row loaded, scores done, value page present.  Stage
   stamps older than t_ready were left by an earlier instruction (an empty
   attention chunk records none). */
MK_API int mk_read_trace(mk_plan_t plan, uint64_t *trace);

MK_API int mk_debug_buffers(mk_plan_t plan, mk_debug_buffers_t *out);

/* Zero counters, queue, epoch, execution counts and the status word. */
MK_API int mk_reset(mk_plan_t plan, void *stream);

/* Free everything the plan owns (synchronises the device first). NULL is a no-op. */
MK_API void mk_destroy(mk_plan_t plan);

/* Grouped-query decode attention that allocates no device memory (the pages
   have no counterpart: this exists for callers that cannot allocate, e.g. a
   serving engine whose device memory is all owned and budgeted by its own
   allocator, or a latency-critical decode loop that must not pay for a
   cudaMalloc).  It needs no plan.  For every sequence b and KV group g it
   computes, for the q heads of that group, softmax(q . k_j / sqrt(d)) . v_j
   over positions j = 0..positions[b] -- the megakernel's attention step,
   split over KV chunks and merged by log-sum-exp.
     q          device fp32 [B][n_q_heads][d]   (already rotated)
     k_cache    device bf16 [B][n_kv_heads][max_ctx][d]  (one layer of the
     v_cache    cache layout of mk_kv_cache, i.e. k + l*B*nkv*max_ctx*d)
     positions  device int32 [B]; an out-of-range position yields NaN rows
     out        device fp32 [B][n_q_heads * d]
   The chunk partials live in one fixed 4 MiB static device array of the
   library (1,048,576 floats; every GPU that loads the library holds it
   until exit); B * n_kv_heads * nchunk * (2*qpg + qpg*d) floats must fit,
   where nchunk = ceil(max_ctx / chunk), chunk = the power of two in 64..256
   nearest above max_ctx/16, else MK_ERR_ARG (nothing launched).  The first
   call on a device resolves the array's device address (once per device,
   with that device current); make that first call before any stream
   capture.  All calls share the array: calls that overlap on the GPU race.
   Asynchronous on `stream`; calls no allocating routine.  Errors: MK_ERR_ARG
   (NULL pointer, unsupported shape, too large for the scratch),
   MK_ERR_DEVICE, MK_ERR_CUDA (also: a CUDA error was already pending when
   the call began; it is left pending for the caller and nothing is
   launched), MK_ERR_LAUNCH (a launch was rejected; a rejected first launch
   queues nothing after it). */
MK_API int mk_attention_noalloc(const float *q, const void *k_cache, const void *v_cache,
                                const int32_t *positions, float *out, int32_t batch,
                                int32_t n_q_heads, int32_t n_kv_heads, int32_t head_dim,
                                int32_t max_ctx, void *stream);

#ifdef __cplusplus
}
#endif
#endif /* MK_H */
