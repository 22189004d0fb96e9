// mk_plan.h -- host planner: instruction list, counters, phases, static
// lists, weight-arena layout and shared-memory layout.
#pragma once
#include <stdint.h>

#include <vector>

#include "mk_internal.h"

namespace mk {

struct HostPlan {
  mk_config cfg{};
  uint32_t num_sms = 0, smem_limit = 0;
  std::vector<mk_instr> instr;
  std::vector<uint32_t> ctr_inc;
  std::vector<mk_phase> phases;
  std::vector<uint32_t> att_first;  // per layer: first instruction of its attention phase
  uint32_t att_count = 0;           // attention instructions per layer
  std::vector<uint32_t> list_off, list_idx;
  std::vector<int32_t> qkv_map;  // permuted q/k/v row -> row of [Wq; Wk; Wv]
  std::vector<int32_t> gu_map;   // gate/up tile row -> row of [Wg; Wu]
  OpGeom geom[8]{};
  std::vector<uint32_t> tiles[8];    // per op: outputs of each tile (QKV: of one group)
  std::vector<uint64_t> rowtab[8];   // per op: arena row -> tile byte offset | row in tile
  uint64_t block_bytes[8]{};         // per op: arena bytes of one layer's block
  // weight arena (bytes)
  std::vector<uint64_t> off_qkv, off_o, off_gu, off_d;
  uint64_t off_lm = 0, off_norms = 0, off_embed = 0, arena_bytes = 0, weight_bytes = 0;
  bool embed_alias = false;  // embedding rows read from the LM-head block
  uint32_t n_wait = 0, n_ctr = 0, lm_ctr = 0;
  uint32_t attn_chunk = 0, nchunk = 0, att_lmax = 0;
  bool tc = false;              // batch > 1: projections on tcgen05, split along K
  bool fp8 = false;             // batch 1: FP8 weight codes, one scale per tile row after
                                // the tile's pages
  std::vector<uint64_t> scaletab[8];  // FP8 plans, per op: arena row -> byte offset of its
                                      // scale in the op's block
  bool stream = false;          // batch 1: every compute warp streams its own weights
  uint32_t tmem_cols = 32;      // tensor-core plans: tensor-memory columns allocated
  bool att_grp = false;         // tensor-core plans, d = 64, <= 4 heads per group: every
                                // attention warp serves all heads of the group
  uint32_t wnb = 0;             // stream plans: ring slots (512 B) per compute warp
  uint32_t tc_nb = 0;           // MMA N: 2 x batch (value and remainder) rounded up to 16
  uint64_t gpart_floats = 0;    // partial-sum buffer of split projections
  uint32_t gemv_arr_base = 0;   // arrival counters of split row blocks
  // shared-memory layout
  uint32_t ring_pages = 0, page_bytes = 0, res_floats = 0;
  uint32_t off_bars = 0, off_fifo = 0, off_meta = 0, off_res = 0, off_att = 0, off_sat = 0,
           off_pos = 0, off_rope = 0, off_normr = 0, off_misc = 0, off_rbuf = 0, off_xs = 0, off_wring = 0, off_deal = 0,
           off_wsc = 0,
           smem_total = 0;
  uint32_t fault_instr = 0xFFFFFFFFu;
};

// Counter ids: waited counters first (compact, cached in shared memory),
// then attention arrival counters, then the LM-head counter.
inline uint32_t ctr_qkv(const mk_config &c, int l, int g) { return l * (c.n_kv_heads + 4) + g; }
inline uint32_t ctr_attn(const mk_config &c, int l) { return l * (c.n_kv_heads + 4) + c.n_kv_heads; }
inline uint32_t ctr_o(const mk_config &c, int l) { return ctr_attn(c, l) + 1; }
inline uint32_t ctr_gu(const mk_config &c, int l) { return ctr_attn(c, l) + 2; }
inline uint32_t ctr_d(const mk_config &c, int l) { return ctr_attn(c, l) + 3; }

// Returns MK_OK or MK_ERR_CONFIG with *why set to a static message.
int build_plan(const mk_config &cfg, uint32_t num_sms, uint32_t smem_limit, HostPlan &P,
               const char **why);

}  // namespace mk
