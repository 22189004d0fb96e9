// mk_runtime.cu -- host side of libmk.so: the C ABI declared in mk.h.
// Device memory, table upload, weight re-tiling, launches, status.
#include <cuda_runtime.h>
#include <math.h>
#include <string.h>

#include <algorithm>
#include <new>
#include <vector>

#include "mk.h"
#include "mk_internal.h"
#include "mk_plan.h"

using namespace mk;

struct mk_plan_s {
  HostPlan H;
  bool host_only = false;
  int device = -1;
  uint8_t *d_arena = nullptr;
  mk_instr *d_instr = nullptr;
  uint32_t *d_aq = nullptr;  // hybrid schedule: per-layer attention queues, first instructions
  uint32_t *d_list_off = nullptr, *d_list_idx = nullptr, *d_ctr = nullptr, *d_ctrl = nullptr,
           *d_exec = nullptr, *d_ctr_inc = nullptr;
  unsigned long long *d_trace = nullptr;
  float *d_x = nullptr, *d_q = nullptr, *d_attn = nullptr, *d_h = nullptr, *d_part = nullptr,
        *d_cos = nullptr, *d_sin = nullptr, *d_logits_stage = nullptr, *d_gpart = nullptr;
  int32_t *d_tok_stage = nullptr, *d_pos_stage = nullptr, *d_qkv_map = nullptr,
          *d_gu_map = nullptr;
  bool weights_loaded = false;
  KParams base{};
  cudaGraphExec_t graph = nullptr;
  const void *graph_key[6] = {};
};

static int cuda_code(cudaError_t e) {
  if (e == cudaSuccess) return MK_OK;
  if (e == cudaErrorMemoryAllocation) return MK_ERR_NOMEM;
  return MK_ERR_CUDA;
}

#define CK(call)                       \
  do {                                 \
    cudaError_t e_ = (call);           \
    if (e_ != cudaSuccess) {           \
      (void)cudaGetLastError();        \
      return cuda_code(e_);            \
    }                                  \
  } while (0)

template <typename T>
static int dalloc(T **ptr, size_t count) {
  cudaError_t e = cudaMalloc((void **)ptr, count * sizeof(T) + 16);
  if (e != cudaSuccess) {
    *ptr = nullptr;
    (void)cudaGetLastError();
    return MK_ERR_NOMEM;
  }
  return MK_OK;
}

extern "C" {

MK_API const char *mk_error_string(int code) {
  switch (code) {
    case MK_OK: return "ok";
    case MK_ERR_CONFIG: return "configuration cannot be planned";
    case MK_ERR_ARG: return "invalid argument";
    case MK_ERR_DEVICE: return "no usable sm_103 device";
    case MK_ERR_NOMEM: return "out of memory";
    case MK_ERR_STATE: return "call out of order";
    case MK_ERR_TIMEOUT: return "device wait exceeded its limit";
    case MK_ERR_BOUNDS: return "token or position out of range";
    case MK_ERR_LAUNCH: return "kernel launch rejected";
    case MK_ERR_CUDA: return "CUDA runtime error";
    default: return "unknown error";
  }
}

static void free_device(mk_plan_s *p) {
  if (p->graph) cudaGraphExecDestroy(p->graph);
  void *ptrs[] = {p->d_aq, p->d_arena, p->d_instr, p->d_list_off, p->d_list_idx, p->d_ctr,
                  p->d_ctrl, p->d_exec, p->d_ctr_inc, p->d_trace, p->d_x,
                  p->d_q, p->d_attn, p->d_h, p->d_part, p->d_cos,
                  p->d_sin, p->d_logits_stage, p->d_tok_stage, p->d_pos_stage, p->d_qkv_map,
                  p->d_gu_map, p->d_gpart};
  for (void *q : ptrs)
    if (q) cudaFree(q);
}

MK_API void mk_destroy(mk_plan_t p) {
  if (!p) return;
  if (!p->host_only) {
    cudaSetDevice(p->device);
    cudaDeviceSynchronize();
    free_device(p);
  }
  delete p;
}

static int setup_device(mk_plan_s *p) {
  const HostPlan &H = p->H;
  const mk_config &c = H.cfg;
  const size_t N = H.instr.size();
  const int B = c.batch, d = c.head_dim;
  const size_t PS = (size_t)2 * (c.n_q_heads / c.n_kv_heads) +
                    (size_t)(c.n_q_heads / c.n_kv_heads) * d;
  int rc = MK_OK;
#define AL(ptr, n)                      \
  if ((rc = dalloc(&(ptr), (n))) != MK_OK) return rc;
  AL(p->d_arena, H.arena_bytes);
  AL(p->d_instr, N);
  AL(p->d_list_off, H.list_off.size());
  AL(p->d_list_idx, H.list_idx.size());
  AL(p->d_aq, (size_t)2 * c.n_layers);  // attention queues, then their first instructions
  AL(p->d_ctr, (size_t)H.n_ctr * kCtrStride);
  AL(p->d_ctrl, (size_t)kCtlWords);
  AL(p->d_exec, N);
  AL(p->d_ctr_inc, (size_t)H.n_ctr);
  if (c.flags & MK_FLAG_TRACE) AL(p->d_trace, N * kTraceWords);
  AL(p->d_x, (size_t)B * c.hidden);
  AL(p->d_q, (size_t)B * c.n_q_heads * d);
  AL(p->d_attn, (size_t)B * c.n_q_heads * d);
  AL(p->d_h, (size_t)B * c.ffn_dim);
  AL(p->d_part, (size_t)B * c.n_kv_heads * H.nchunk * PS);
  AL(p->d_cos, (size_t)c.max_ctx * (d / 2));
  AL(p->d_sin, (size_t)c.max_ctx * (d / 2));
  AL(p->d_logits_stage, (size_t)B * c.vocab);
  AL(p->d_tok_stage, (size_t)B);
  AL(p->d_pos_stage, (size_t)B);
  AL(p->d_qkv_map, H.qkv_map.size());
  AL(p->d_gu_map, H.gu_map.size());
  if (H.tc) AL(p->d_gpart, H.gpart_floats);
#undef AL
  CK(cudaMemcpy(p->d_instr, H.instr.data(), N * sizeof(mk_instr), cudaMemcpyHostToDevice));
  CK(cudaMemcpy(p->d_list_off, H.list_off.data(), H.list_off.size() * 4, cudaMemcpyHostToDevice));
  CK(cudaMemcpy(p->d_list_idx, H.list_idx.data(), H.list_idx.size() * 4, cudaMemcpyHostToDevice));
  CK(cudaMemset(p->d_aq, 0, (size_t)c.n_layers * 4));
  CK(cudaMemcpy(p->d_aq + c.n_layers, H.att_first.data(), (size_t)c.n_layers * 4,
                cudaMemcpyHostToDevice));
  CK(cudaMemcpy(p->d_ctr_inc, H.ctr_inc.data(), H.n_ctr * 4, cudaMemcpyHostToDevice));
  CK(cudaMemcpy(p->d_qkv_map, H.qkv_map.data(), H.qkv_map.size() * 4, cudaMemcpyHostToDevice));
  CK(cudaMemcpy(p->d_gu_map, H.gu_map.data(), H.gu_map.size() * 4, cudaMemcpyHostToDevice));
  CK(cudaMemset(p->d_ctr, 0, (size_t)H.n_ctr * kCtrStride * 4));
  CK(cudaMemset(p->d_ctrl, 0, (size_t)kCtlWords * 4));
  CK(cudaMemset(p->d_exec, 0, N * 4));
  CK(cudaMemset(p->d_x, 0, (size_t)B * c.hidden * 4));
  // RoPE table: angle p * theta^(-2i/d) in double, stored as fp32 cos / sin
  {
    const int half = d / 2;
    std::vector<float> cs((size_t)c.max_ctx * half), sn((size_t)c.max_ctx * half);
    for (int pos = 0; pos < c.max_ctx; ++pos)
      for (int i = 0; i < half; ++i) {
        const double inv = pow((double)c.rope_theta, -2.0 * i / d);
        const double a = (double)pos * inv;
        cs[(size_t)pos * half + i] = (float)cos(a);
        sn[(size_t)pos * half + i] = (float)sin(a);
      }
    CK(cudaMemcpy(p->d_cos, cs.data(), cs.size() * 4, cudaMemcpyHostToDevice));
    CK(cudaMemcpy(p->d_sin, sn.data(), sn.size() * 4, cudaMemcpyHostToDevice));
  }
  CK(H.stream ? set_stream_smem(H.smem_total) : set_megakernel_smem(H.smem_total));

  KParams &P = p->base;
  memset(&P, 0, sizeof P);
  P.instr = p->d_instr;
  P.n_instr = (uint32_t)N;
  P.list_off = p->d_list_off;
  P.list_idx = p->d_list_idx;
  P.aq = p->d_aq;
  P.att_first = p->d_aq + c.n_layers;
  P.att_count = H.att_count;
  P.ctr = p->d_ctr;
  P.ctrl = p->d_ctrl;
  P.exec = p->d_exec;
  P.ctr_inc = p->d_ctr_inc;
  P.trace = p->d_trace;
  P.arena = p->d_arena;
  P.embed = reinterpret_cast<const uint16_t *>(p->d_arena + (H.embed_alias ? H.off_lm : H.off_embed));
  P.norms = reinterpret_cast<const uint16_t *>(p->d_arena + H.off_norms);
  P.x = p->d_x;
  P.q = p->d_q;
  P.attn = p->d_attn;
  P.h = p->d_h;
  P.part = p->d_part;
  P.rope_cos = p->d_cos;
  P.rope_sin = p->d_sin;
  for (int i = 0; i < 8; ++i) P.geom[i] = H.geom[i];
  P.L = c.n_layers;
  P.H = c.hidden;
  P.nq = c.n_q_heads;
  P.nkv = c.n_kv_heads;
  P.d = d;
  P.F = c.ffn_dim;
  P.V = c.vocab;
  P.B = B;
  P.max_ctx = c.max_ctx;
  P.qpg = c.n_q_heads / c.n_kv_heads;
  P.nchunk = (int32_t)H.nchunk;
  P.attn_chunk = (int32_t)H.attn_chunk;
  P.att_lmax = (int32_t)H.att_lmax;
  P.tc = H.tc ? 1 : 0;
  P.tc_nb = (int32_t)H.tc_nb;
  P.stream = H.stream ? 1 : 0;
  P.att_grp = H.att_grp ? 1 : 0;
  P.fp8 = H.fp8 ? 1 : 0;
  P.tmem_cols = H.tmem_cols;
  P.wnb = H.wnb;
  P.off_wring = H.off_wring;
  P.gpart = p->d_gpart;
  P.eps = c.rms_eps;
  P.attn_scale = (float)(1.0 / sqrt((double)d));
  P.n_wait = (int32_t)H.n_wait;
  P.mode = c.sched_mode == MK_SCHED_STATIC   ? kModeStatic
           : c.sched_mode == MK_SCHED_HYBRID ? kModeHybrid
                                             : kModeDynamic;
  P.n_blocks = H.num_sms;
  P.flags = c.flags;
  // wait limits count SM cycles; budget them at the maximum SM clock
  int clk_khz = 2100000;
  if (cudaDeviceGetAttribute(&clk_khz, cudaDevAttrClockRate, p->device) != cudaSuccess || clk_khz <= 0) {
    (void)cudaGetLastError();
    clk_khz = 2100000;
  }
  P.timeout_cycles = (uint64_t)(c.wait_timeout_us > 0 ? c.wait_timeout_us : 1000000) * (uint64_t)clk_khz / 1000ull;
  // static lists may run a full FIFO ahead; the dynamic queue claims close
  // to need so the claims still balance the blocks
  P.lookahead = P.mode == kModeDynamic ? 3u : (uint32_t)kFifo;
  P.loader_idle_ns = 64;
  P.l2_window = c.l2_prefetch_kb > 0 ? (uint32_t)c.l2_prefetch_kb * 1024u : 0u;
  P.ring_pages = H.ring_pages;
  P.page_bytes = H.page_bytes;
  P.off_bars = H.off_bars;
  P.off_fifo = H.off_fifo;
  P.off_meta = H.off_meta;
  P.off_res = H.off_res;
  P.res_floats = H.res_floats;
  P.off_att = H.off_att;
  P.off_sat = H.off_sat;
  P.off_pos = H.off_pos;
  P.off_rope = H.off_rope;
  P.off_normr = H.off_normr;
  P.off_misc = H.off_misc;
  P.off_deal = H.off_deal;
  P.off_rbuf = H.off_rbuf;
  P.off_xs = H.off_xs;
  P.off_wsc = H.off_wsc;
  P.smem_total = H.smem_total;
  return MK_OK;
}

MK_API int mk_plan(const mk_config *cfg, mk_plan_t *out) {
  if (!cfg || !out) return MK_ERR_ARG;
  *out = nullptr;
  mk_plan_s *p = new (std::nothrow) mk_plan_s();
  if (!p) return MK_ERR_NOMEM;
  p->host_only = (cfg->flags & MK_FLAG_HOST_ONLY) != 0;
  uint32_t sms = 0, smem = 0;
  if (p->host_only) {
    if (cfg->num_sms <= 0) {
      delete p;
      return MK_ERR_ARG;
    }
    sms = (uint32_t)cfg->num_sms;
    smem = cfg->smem_bytes > 0 ? (uint32_t)cfg->smem_bytes : 232448u;
  } else {
    int dev = 0, major = 0, minor = 0, nsm = 0, optin = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) !=
            cudaSuccess) {
      (void)cudaGetLastError();
      delete p;
      return MK_ERR_DEVICE;
    }
    if (major != 10 || minor != 3) {  // the library carries sm_103a code only
      delete p;
      return MK_ERR_DEVICE;
    }
    p->device = dev;
    sms = cfg->num_sms > 0 && cfg->num_sms < nsm ? (uint32_t)cfg->num_sms : (uint32_t)nsm;
    smem = cfg->smem_bytes > 0 && cfg->smem_bytes < optin ? (uint32_t)cfg->smem_bytes
                                                           : (uint32_t)optin;
  }
  const char *why = nullptr;
  int rc = build_plan(*cfg, sms, smem, p->H, &why);
  if (rc != MK_OK) {
    delete p;
    return rc;
  }
  if (!p->host_only) {
    rc = setup_device(p);
    if (rc != MK_OK) {
      free_device(p);
      delete p;
      return rc;
    }
  }
  *out = p;
  return MK_OK;
}

MK_API int mk_plan_info(mk_plan_t p, mk_plan_info_t *info) {
  if (!p || !info) return MK_ERR_ARG;
  const HostPlan &H = p->H;
  memset(info, 0, sizeof *info);
  info->n_instr = (uint32_t)H.instr.size();
  info->n_counters = H.n_ctr;
  info->n_wait_counters = H.n_wait;
  info->n_phases = (uint32_t)H.phases.size();
  info->n_blocks = H.num_sms;
  info->threads = kThreads;
  info->ring_pages = H.ring_pages;
  info->page_bytes = H.page_bytes;
  info->fifo_depth = kFifo;
  info->smem_bytes = H.smem_total;
  info->attn_nchunk = H.nchunk;
  info->attn_chunk = H.attn_chunk;
  info->arena_bytes = H.arena_bytes;
  info->weight_bytes = H.weight_bytes;
  info->warp_ring_slots = H.stream ? H.wnb : 0u;
  info->kernel = H.stream ? 2u : H.tc ? 1u : H.fp8 ? 3u : 0u;
  return MK_OK;
}

MK_API int mk_plan_tables(mk_plan_t p, const mk_instr **instr, size_t *n_instr,
                          const uint32_t **counter_inc, size_t *n_counters) {
  if (!p) return MK_ERR_ARG;
  if (instr) *instr = p->H.instr.data();
  if (n_instr) *n_instr = p->H.instr.size();
  if (counter_inc) *counter_inc = p->H.ctr_inc.data();
  if (n_counters) *n_counters = p->H.n_ctr;
  return MK_OK;
}

MK_API int mk_plan_phases(mk_plan_t p, const mk_phase **phases, size_t *n_phases) {
  if (!p) return MK_ERR_ARG;
  if (phases) *phases = p->H.phases.data();
  if (n_phases) *n_phases = p->H.phases.size();
  return MK_OK;
}

MK_API int mk_plan_lists(mk_plan_t p, const uint32_t **list_off, const uint32_t **list_idx,
                         size_t *n_lists) {
  if (!p) return MK_ERR_ARG;
  if (list_off) *list_off = p->H.list_off.data();
  if (list_idx) *list_idx = p->H.list_idx.data();
  if (n_lists) *n_lists = p->H.num_sms;
  return MK_OK;
}

// ---- weights ----------------------------------------------------------------
static int copy_in(void *dst, const void *src, size_t bytes, cudaStream_t s) {
  if (!src) return MK_ERR_ARG;
  CK(cudaMemcpyAsync(dst, src, bytes, cudaMemcpyDefault, s));
  return MK_OK;
}

MK_API int mk_load_weights(mk_plan_t p, const mk_weights *w, void *stream) {
  if (!p || !w || !w->embed || !w->final_norm || !w->layers) return MK_ERR_ARG;
  if (p->host_only) return MK_ERR_STATE;
  const HostPlan &H = p->H;
  const mk_config &c = H.cfg;
  if (!c.tie_embeddings && !w->lm_head) return MK_ERR_ARG;
  for (int l = 0; l < c.n_layers; ++l) {
    const mk_layer_weights &lw = w->layers[l];
    if (!lw.attn_norm || !lw.wq || !lw.wk || !lw.wv || !lw.wo || !lw.mlp_norm || !lw.w_gate ||
        !lw.w_up || !lw.w_down)
      return MK_ERR_ARG;
  }
  CK(cudaSetDevice(p->device));
  cudaStream_t s = (cudaStream_t)stream;
  const size_t H_ = c.hidden, F = c.ffn_dim, V = c.vocab, QD = (size_t)c.n_q_heads * c.head_dim,
               KD = (size_t)c.n_kv_heads * c.head_dim;
  size_t stage_elems = (QD + 2 * KD) * H_;
  stage_elems = std::max(stage_elems, 2 * F * H_);
  stage_elems = std::max(stage_elems, H_ * QD);
  stage_elems = std::max(stage_elems, V * H_);
  uint8_t *stage = nullptr;
  if (dalloc(&stage, stage_elems * 2) != MK_OK) return MK_ERR_NOMEM;
  // the planner's row tables (arena row -> tile offset | row in tile), one per op,
  // and for FP8 plans, after them, the row-scale tables (arena row -> scale offset)
  size_t rt_rows = 0, rt_at[8] = {};
  for (int op = MK_OP_QKV; op <= MK_OP_LMHEAD; ++op) {
    rt_at[op] = rt_rows;
    rt_rows += H.rowtab[op].size();
  }
  uint64_t *rowtab = nullptr;
  if (dalloc(&rowtab, H.fp8 ? 2 * rt_rows : rt_rows) != MK_OK) {
    cudaFree(stage);
    return MK_ERR_NOMEM;
  }
  uint64_t *scaletab = rowtab + rt_rows;
  int rc = MK_OK;
  for (int op = MK_OP_QKV; op <= MK_OP_LMHEAD && rc == MK_OK; ++op) {
    if (!H.rowtab[op].empty() &&
        cudaMemcpy(rowtab + rt_at[op], H.rowtab[op].data(), H.rowtab[op].size() * 8,
                   cudaMemcpyHostToDevice) != cudaSuccess) {
      (void)cudaGetLastError();
      rc = MK_ERR_CUDA;
    }
    if (H.fp8 && rc == MK_OK &&
        (H.scaletab[op].size() != H.rowtab[op].size() ||
         cudaMemcpy(scaletab + rt_at[op], H.scaletab[op].data(), H.scaletab[op].size() * 8,
                    cudaMemcpyHostToDevice) != cudaSuccess)) {
      (void)cudaGetLastError();
      rc = MK_ERR_CUDA;
    }
  }
  const uint32_t pg = H.page_bytes;
  uint8_t *A = p->d_arena;
  auto norm_dst = [&](int idx) { return A + H.off_norms + (size_t)idx * H_ * 2; };
  auto retile = [&](uint8_t *dst, const int32_t *map, uint32_t rows, int op) {
    cudaError_t e;
    if (H.tc) {
      e = launch_retile_tc(dst, stage, map, rows, H.geom[op], pg, s);
    } else if (H.stream) {
      if (rows != H.rowtab[op].size()) return MK_ERR_CONFIG;
      e = launch_retile_stream(dst, stage, map, rowtab + rt_at[op], rows, H.geom[op], s);
    } else if (H.fp8) {  // row scales first, then the codes (same stream)
      if (rows != H.rowtab[op].size()) return MK_ERR_CONFIG;
      e = launch_row_scale(dst, stage, map, scaletab + rt_at[op], rows, H.geom[op].K, s);
      if (e == cudaSuccess)
        e = launch_retile_q8(dst, stage, map, rowtab + rt_at[op], scaletab + rt_at[op], rows,
                             H.geom[op], pg, s);
    } else {
      if (rows != H.rowtab[op].size()) return MK_ERR_CONFIG;
      e = launch_retile(dst, stage, map, rowtab + rt_at[op], rows, H.geom[op], pg, s);
    }
    return e == cudaSuccess ? MK_OK : cuda_code(e);
  };
#define TRY(x)                  \
  if ((rc = (x)) != MK_OK) {    \
    (void)cudaGetLastError();   \
    goto done;                  \
  }
  TRY(rc);
  for (int l = 0; l < c.n_layers; ++l) {
    const mk_layer_weights &lw = w->layers[l];
    TRY(copy_in(norm_dst(2 * l), lw.attn_norm, H_ * 2, s));
    TRY(copy_in(norm_dst(2 * l + 1), lw.mlp_norm, H_ * 2, s));
    TRY(copy_in(stage, lw.wq, QD * H_ * 2, s));
    TRY(copy_in(stage + QD * H_ * 2, lw.wk, KD * H_ * 2, s));
    TRY(copy_in(stage + (QD + KD) * H_ * 2, lw.wv, KD * H_ * 2, s));
    TRY(retile(A + H.off_qkv[l], p->d_qkv_map, (uint32_t)(QD + 2 * KD), MK_OP_QKV));
    TRY(copy_in(stage, lw.wo, H_ * QD * 2, s));
    TRY(retile(A + H.off_o[l], nullptr, (uint32_t)H_, MK_OP_OPROJ));
    TRY(copy_in(stage, lw.w_gate, F * H_ * 2, s));
    TRY(copy_in(stage + F * H_ * 2, lw.w_up, F * H_ * 2, s));
    TRY(retile(A + H.off_gu[l], p->d_gu_map, (uint32_t)(2 * F), MK_OP_GATEUP));
    TRY(copy_in(stage, lw.w_down, H_ * F * 2, s));
    TRY(retile(A + H.off_d[l], nullptr, (uint32_t)H_, MK_OP_DOWN));
  }
  TRY(copy_in(norm_dst(2 * c.n_layers), w->final_norm, H_ * 2, s));
  TRY(copy_in(stage, c.tie_embeddings ? w->embed : w->lm_head, V * H_ * 2, s));
  TRY(retile(A + H.off_lm, nullptr, (uint32_t)V, MK_OP_LMHEAD));
  if (!H.embed_alias) TRY(copy_in(A + H.off_embed, w->embed, V * H_ * 2, s));
  if (cudaStreamSynchronize(s) != cudaSuccess) {
    (void)cudaGetLastError();
    rc = MK_ERR_CUDA;
  }
#undef TRY
done:
  cudaStreamSynchronize(s);
  cudaFree(stage);
  cudaFree(rowtab);
  if (rc == MK_OK) p->weights_loaded = true;
  return rc;
}

// ---- steps ------------------------------------------------------------------
static int check_step(mk_plan_t p, const int32_t *tokens, const int32_t *positions,
                      const mk_kv_cache *kv, float *logits) {
  if (!p || !tokens || !positions || !kv || !kv->k || !kv->v || !logits) return MK_ERR_ARG;
  if (p->host_only || !p->weights_loaded) return MK_ERR_STATE;
  return MK_OK;
}

static KParams step_params(mk_plan_t p, const int32_t *tokens, const int32_t *positions,
                           const mk_kv_cache *kv, float *logits) {
  KParams P = p->base;
  P.tokens = tokens;
  P.positions = positions;
  P.kc = static_cast<uint16_t *>(kv->k);
  P.vc = static_cast<uint16_t *>(kv->v);
  P.logits = logits;
  return P;
}

MK_API int mk_decode_step(mk_plan_t p, const int32_t *tokens, const int32_t *positions,
                          const mk_kv_cache *kv, float *logits, void *stream) {
  int rc = check_step(p, tokens, positions, kv, logits);
  if (rc != MK_OK) return rc;
  cudaSetDevice(p->device);
  const KParams P = step_params(p, tokens, positions, kv, logits);
  const cudaError_t le = P.stream ? launch_megakernel_stream(P, p->H.num_sms, true, (cudaStream_t)stream)
                                  : launch_megakernel(P, p->H.num_sms, true, (cudaStream_t)stream);
  if (le != cudaSuccess) {
    (void)cudaGetLastError();
    return MK_ERR_LAUNCH;
  }
  return MK_OK;
}

MK_API int mk_decode_step_host(mk_plan_t p, const int32_t *tokens, const int32_t *positions,
                               const mk_kv_cache *kv, float *logits, void *stream) {
  if (!p || !tokens || !positions || !logits) return MK_ERR_ARG;
  cudaStream_t s = (cudaStream_t)stream;
  const size_t B = p->H.cfg.batch, V = p->H.cfg.vocab;
  if (p->host_only || !p->weights_loaded) return MK_ERR_STATE;
  cudaSetDevice(p->device);
  CK(cudaMemcpyAsync(p->d_tok_stage, tokens, B * 4, cudaMemcpyHostToDevice, s));
  CK(cudaMemcpyAsync(p->d_pos_stage, positions, B * 4, cudaMemcpyHostToDevice, s));
  int rc = mk_decode_step(p, p->d_tok_stage, p->d_pos_stage, kv, p->d_logits_stage, stream);
  if (rc != MK_OK) return rc;
  CK(cudaMemcpyAsync(logits, p->d_logits_stage, B * V * 4, cudaMemcpyDeviceToHost, s));
  CK(cudaStreamSynchronize(s));
  return MK_OK;
}

static int enqueue_phases(mk_plan_t p, const KParams &base, cudaStream_t s, int only_phase) {
  KParams P = base;
  P.mode = kModeRange;
  const size_t nph = p->H.phases.size();
  for (size_t i = 0; i < nph; ++i) {
    if (only_phase >= 0 && (size_t)only_phase != i) continue;
    const mk_phase &ph = p->H.phases[i];
    P.range_first = ph.first;
    P.range_count = ph.count;
    const cudaError_t le = P.stream ? launch_megakernel_stream(P, ph.count, false, s)
                                    : launch_megakernel(P, ph.count, false, s);
    if (le != cudaSuccess) {
      (void)cudaGetLastError();
      return MK_ERR_LAUNCH;
    }
  }
  if (only_phase < 0 && launch_epoch_advance(p->d_ctrl, s) != cudaSuccess) {
    (void)cudaGetLastError();
    return MK_ERR_LAUNCH;
  }
  return MK_OK;
}

MK_API int mk_multikernel_step(mk_plan_t p, const int32_t *tokens, const int32_t *positions,
                               const mk_kv_cache *kv, float *logits, int use_graph,
                               void *stream) {
  int rc = check_step(p, tokens, positions, kv, logits);
  if (rc != MK_OK) return rc;
  cudaSetDevice(p->device);
  cudaStream_t s = (cudaStream_t)stream;
  const KParams P = step_params(p, tokens, positions, kv, logits);
  if (!use_graph) return enqueue_phases(p, P, s, -1);
  const void *key[6] = {tokens, positions, kv->k, kv->v, logits, stream};
  if (!p->graph || memcmp(key, p->graph_key, sizeof key) != 0) {
    if (p->graph) {
      cudaGraphExecDestroy(p->graph);
      p->graph = nullptr;
    }
    cudaStream_t cs;
    CK(cudaStreamCreateWithFlags(&cs, cudaStreamNonBlocking));
    cudaGraph_t g = nullptr;
    if (cudaStreamBeginCapture(cs, cudaStreamCaptureModeThreadLocal) != cudaSuccess) {
      cudaStreamDestroy(cs);
      (void)cudaGetLastError();
      return MK_ERR_CUDA;
    }
    rc = enqueue_phases(p, P, cs, -1);
    cudaError_t e = cudaStreamEndCapture(cs, &g);
    cudaStreamDestroy(cs);
    if (rc != MK_OK || e != cudaSuccess) {
      if (g) cudaGraphDestroy(g);
      (void)cudaGetLastError();
      return rc != MK_OK ? rc : MK_ERR_CUDA;
    }
    e = cudaGraphInstantiate(&p->graph, g, 0);
    cudaGraphDestroy(g);
    if (e != cudaSuccess) {
      p->graph = nullptr;
      (void)cudaGetLastError();
      return MK_ERR_CUDA;
    }
    memcpy(p->graph_key, key, sizeof key);
  }
  CK(cudaGraphLaunch(p->graph, s));
  return MK_OK;
}

MK_API int mk_run_phase(mk_plan_t p, int phase, const int32_t *tokens, const int32_t *positions,
                        const mk_kv_cache *kv, float *logits, void *stream) {
  int rc = check_step(p, tokens, positions, kv, logits);
  if (rc != MK_OK) return rc;
  if (phase < 0 || (size_t)phase >= p->H.phases.size()) return MK_ERR_ARG;
  cudaSetDevice(p->device);
  return enqueue_phases(p, step_params(p, tokens, positions, kv, logits), (cudaStream_t)stream,
                        phase);
}

// ---- status and introspection -------------------------------------------------
static int reset_state(mk_plan_t p, cudaStream_t s) {
  CK(cudaMemsetAsync(p->d_ctr, 0, (size_t)p->H.n_ctr * kCtrStride * 4, s));
  CK(cudaMemsetAsync(p->d_ctrl, 0, (size_t)kCtlWords * 4, s));
  CK(cudaMemsetAsync(p->d_exec, 0, p->H.instr.size() * 4, s));
  CK(cudaMemsetAsync(p->d_aq, 0, (size_t)p->H.cfg.n_layers * 4, s));
  CK(cudaStreamSynchronize(s));
  return MK_OK;
}

MK_API int mk_reset(mk_plan_t p, void *stream) {
  if (!p) return MK_ERR_ARG;
  if (p->host_only) return MK_ERR_STATE;
  cudaSetDevice(p->device);
  return reset_state(p, (cudaStream_t)stream);
}

MK_API int mk_status(mk_plan_t p, void *stream) {
  if (!p) return MK_ERR_ARG;
  if (p->host_only) return MK_ERR_STATE;
  cudaSetDevice(p->device);
  cudaStream_t s = (cudaStream_t)stream;
  CK(cudaStreamSynchronize(s));
  uint32_t ctl[4] = {0, 0, 0, 0};
  CK(cudaMemcpy(ctl, p->d_ctrl, sizeof ctl, cudaMemcpyDeviceToHost));
  int code = (int)ctl[kCtlStatus];
  if (code == 0 && ctl[kCtlAbort]) code = MK_ERR_TIMEOUT;
  if (code != 0) {
    int rc = reset_state(p, s);
    if (rc != MK_OK) return rc;
  }
  return code;
}

MK_API int mk_read_counters(mk_plan_t p, uint32_t *counters, uint32_t *queue, uint32_t *exec,
                            uint32_t *epoch) {
  if (!p) return MK_ERR_ARG;
  if (p->host_only) return MK_ERR_STATE;
  cudaSetDevice(p->device);
  CK(cudaDeviceSynchronize());
  if (counters) {
    std::vector<uint32_t> all((size_t)p->H.n_ctr * kCtrStride);
    CK(cudaMemcpy(all.data(), p->d_ctr, all.size() * 4, cudaMemcpyDeviceToHost));
    for (uint32_t c = 0; c < p->H.n_ctr; ++c) counters[c] = all[(size_t)c * kCtrStride];
  }
  uint32_t ctl[kCtlWords];
  CK(cudaMemcpy(ctl, p->d_ctrl, sizeof ctl, cudaMemcpyDeviceToHost));
  if (queue) *queue = ctl[kCtlQueue];
  if (epoch) *epoch = ctl[kCtlEpoch];
  if (exec) CK(cudaMemcpy(exec, p->d_exec, p->H.instr.size() * 4, cudaMemcpyDeviceToHost));
  return MK_OK;
}

MK_API int mk_read_trace(mk_plan_t p, uint64_t *trace) {
  if (!p || !trace) return MK_ERR_ARG;
  if (p->host_only || !p->d_trace) return MK_ERR_STATE;
  cudaSetDevice(p->device);
  CK(cudaDeviceSynchronize());
  CK(cudaMemcpy(trace, p->d_trace, p->H.instr.size() * kTraceWords * 8, cudaMemcpyDeviceToHost));
  return MK_OK;
}

MK_API int mk_debug_buffers(mk_plan_t p, mk_debug_buffers_t *out) {
  if (!p || !out) return MK_ERR_ARG;
  if (p->host_only) return MK_ERR_STATE;
  out->x = p->d_x;
  out->q = p->d_q;
  out->attn = p->d_attn;
  out->h = p->d_h;
  return MK_OK;
}

}  // extern "C"
