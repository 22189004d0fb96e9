/*
 * replay.c -- TEST INFRASTRUCTURE ONLY.  Independent replay of a megakernel
 * instruction table.  It decodes the table from its documented byte format
 * (64-byte little-endian records; the field offsets are restated below, not
 * taken from the library's header) and checks it against the decoder's data
 * flow, which this file derives on its own from the operations' meaning.
 *
 * The mechanism being checked is the one the pages describe:
 *  - « 2 · Définition et généalogie », §2.6, "3. Les compteurs de dépendance":
 *    a producer makes its data visible, then adds 1 to its output counter; a
 *    consumer waits until its input counter reaches a target value.
 *  - §2.6, "5. L'ordonnancement" and §2.4 (persistent-threads loop): SMs take
 *    instructions from a global queue (atomic counter) or from a per-SM list.
 *  - §2.6 "1. La persistance" and the chapter's questions: counter waits only
 *    make progress if every block is resident; a wait on an instruction that
 *    is later in the queue would be a deadlock.
 *
 * Record layout (bytes): 0 op u8 | 1 flags u8 | 2 layer u16 | 4 b u16 | 6 g u16 |
 *   8 wait_ctr u32 | 12 wait_tgt u32 | 16 sig_ctr u32 | 20 sig2_ctr u32 |
 *   24 sig2_after u32 | 28 row0 u32 | 32 nrows u32 | 36 chunk u32 |
 *   40 nchunk u32 | 44 npages u32 | 48 wofs u64 | 56 phase u32 | 60 reserved u32.
 * Ops: 1 RMSNorm+QKV+RoPE, 2 attention chunk, 3 O-projection, 4 RMSNorm+gate/up,
 *   5 down-projection, 6 final norm + LM head.  Counter id 0xFFFFFFFF = none.
 * Output rows: op 1 -> rows of the fused q/k/v output, grouped per KV head
 *   (q heads of the group, then its k head, then its v head); op 4 -> FFN
 *   activations h; ops 3, 5 -> residual rows; op 6 -> vocabulary rows.
 * An attention chunk adds 1 to its group's arrival counter; the chunk that
 *   brings that counter to sig2_after for the step (the last of the group)
 *   merges the group and adds 1 to sig2_ctr.  A projection may be split the
 *   same way along its input dimension (batch > 1 plans): the slices of one
 *   block of output rows (same op, layer and row0; chunk = slice index,
 *   nchunk = slices) each add 1 to the block's arrival counter, and the last
 *   one sums the slices, writes the rows and adds 1 to sig2_ctr.
 */
#include <stdarg.h>
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include "oracle.h"

#define NONE 0xFFFFFFFFu
enum { OQKV = 1, OATTN = 2, OOPROJ = 3, OGATEUP = 4, ODOWN = 5, OLM = 6 };

typedef struct {
  int op, flags, layer, b, g;
  uint32_t wait_ctr, wait_tgt, sig_ctr, sig2_ctr, sig2_after, row0, nrows, chunk, nchunk;
} rec_t;

static uint32_t u32_at(const uint8_t *p, int off) {
  uint32_t v;
  memcpy(&v, p + off, 4);
  return v;
}
static uint32_t u16_at(const uint8_t *p, int off) {
  uint16_t v;
  memcpy(&v, p + off, 2);
  return v;
}

static void decode(const void *table, int i, rec_t *r) {
  const uint8_t *p = (const uint8_t *)table + (size_t)i * 64;
  r->op = p[0];
  r->flags = p[1];
  r->layer = (int)u16_at(p, 2);
  r->b = (int)u16_at(p, 4);
  r->g = (int)u16_at(p, 6);
  r->wait_ctr = u32_at(p, 8);
  r->wait_tgt = u32_at(p, 12);
  r->sig_ctr = u32_at(p, 16);
  r->sig2_ctr = u32_at(p, 20);
  r->sig2_after = u32_at(p, 24);
  r->row0 = u32_at(p, 28);
  r->nrows = u32_at(p, 32);
  r->chunk = u32_at(p, 36);
  r->nchunk = u32_at(p, 40);
}

static int fail(char *msg, int len, const char *fmt, ...) {
  if (msg && len > 0) {
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(msg, (size_t)len, fmt, ap);
    va_end(ap);
  }
  return -1;
}

/* ---- small growable int lists --------------------------------------------- */
typedef struct {
  int *v;
  int n, cap;
} ilist;
static void push(ilist *l, int x) {
  if (l->n == l->cap) {
    l->cap = l->cap ? 2 * l->cap : 8;
    l->v = (int *)realloc(l->v, sizeof(int) * (size_t)l->cap);
  }
  l->v[l->n++] = x;
}
static void free_lists(ilist *ls, int n) {
  if (!ls) return;
  for (int i = 0; i < n; ++i) free(ls[i].v);
  free(ls);
}

/* ---- replay --------------------------------------------------------------- */
typedef struct {
  int N, M, n_ctr, words;
  rec_t *r;
  ilist *events;   /* per counter: nodes whose completion adds 1 to it */
  ilist *chunks;   /* per merge node: its chunk instructions */
  uint64_t **clo;  /* per counter: closure bitset (lazy) */
  int *state;      /* per counter: 0 not computed, 1 in progress, 2 done */
  int cycle;
} ctx_t;

static int merge_id(const or_shape *s, int l, int b, int g) {
  return (l * s->B + b) * s->nkv + g;
}

static uint64_t *closure_of_ctr(ctx_t *c, uint32_t ctr);

/* closure of a node: every node that has completed before it may start */
static void or_node_closure(ctx_t *c, int node, uint64_t *acc) {
  if (node < c->N) {
    uint32_t w = c->r[node].wait_ctr;
    if (w == NONE) return;
    uint64_t *cl = closure_of_ctr(c, w);
    if (!cl) return;
    for (int k = 0; k < c->words; ++k) acc[k] |= cl[k];
  } else {
    ilist *ch = &c->chunks[node - c->N];
    for (int j = 0; j < ch->n; ++j) {
      int x = ch->v[j];
      acc[x >> 6] |= 1ull << (x & 63);
      or_node_closure(c, x, acc);
    }
  }
}

static uint64_t *closure_of_ctr(ctx_t *c, uint32_t ctr) {
  if (ctr >= (uint32_t)c->n_ctr) return 0;
  if (c->state[ctr] == 2) return c->clo[ctr];
  if (c->state[ctr] == 1) {
    c->cycle = 1;
    return 0;
  }
  c->state[ctr] = 1;
  uint64_t *acc = (uint64_t *)calloc((size_t)c->words, 8);
  ilist *ev = &c->events[ctr];
  /* group instruction events by their own wait so each closure is ORed once */
  uint32_t last_wait = NONE - 1;
  for (int j = 0; j < ev->n; ++j) {
    int x = ev->v[j];
    acc[x >> 6] |= 1ull << (x & 63);
    if (x < c->N) {
      if (c->r[x].wait_ctr == last_wait) continue;
      last_wait = c->r[x].wait_ctr;
    }
    or_node_closure(c, x, acc);
  }
  c->clo[ctr] = acc;
  c->state[ctr] = 2;
  return acc;
}

static int has(const uint64_t *bits, int x) { return (int)((bits[x >> 6] >> (x & 63)) & 1u); }

int or_replay(const void *table, int N, int n_ctr, const or_shape *s, int S,
              const uint32_t *list_off, const uint32_t *list_idx, uint32_t *inc_out, char *msg,
              int msg_len) {
  if (!table || N <= 0 || n_ctr <= 0 || !s) return fail(msg, msg_len, "bad arguments");
  const int L = s->L, B = s->B, nkv = s->nkv, nq = s->nq, d = s->d;
  if (nq % nkv) return fail(msg, msg_len, "nq %% nkv != 0");
  const int qpg = nq / nkv;
  const int QKV_ROWS = (nq + 2 * nkv) * d, GROUP_ROWS = (qpg + 2) * d;
  int rc = 0;
  ctx_t c;
  memset(&c, 0, sizeof c);
  c.N = N;
  const int M_att = L * B * nkv;  /* attention groups first, then split projections */
  c.M = M_att + N;
  c.n_ctr = n_ctr;
  c.words = (N + c.M + 63) / 64;
  c.r = (rec_t *)calloc((size_t)N, sizeof(rec_t));
  c.events = (ilist *)calloc((size_t)n_ctr, sizeof(ilist));
  c.chunks = (ilist *)calloc((size_t)c.M, sizeof(ilist));
  c.clo = (uint64_t **)calloc((size_t)n_ctr, sizeof(uint64_t *));
  c.state = (int *)calloc((size_t)n_ctr, sizeof(int));
  /* per (op, layer) instruction lists; qkv per (l,g) */
  ilist *byop = (ilist *)calloc((size_t)7 * (L + 1), sizeof(ilist));
  ilist *qkv_g = (ilist *)calloc((size_t)L * nkv, sizeof(ilist));
  unsigned char *cov_qkv = 0, *cov_h = 0, *cov_x3 = 0, *cov_x5 = 0, *cov_lm = 0, *cov_att = 0;
  uint32_t *nchunk_of = (uint32_t *)calloc((size_t)c.M, sizeof(uint32_t));
  /* split projections: (op, layer, row0) -> group id, open addressing */
  const size_t hcap = 2 * (size_t)N + 1;
  uint64_t *hkey = (uint64_t *)calloc(hcap, sizeof(uint64_t));
  int *hval = (int *)calloc(hcap, sizeof(int));
  int n_split = 0;
#define BYOP(op, l) byop[(op) * (L + 1) + (l)]

  /* 1. decode + field checks */
  for (int i = 0; i < N; ++i) {
    rec_t *r = &c.r[i];
    decode(table, i, r);
    if (r->op < OQKV || r->op > OLM) {
      rc = fail(msg, msg_len, "instr %d: bad op %d", i, r->op);
      goto out;
    }
    int lmax = r->op == OLM ? 1 : L;
    if (r->layer < 0 || r->layer >= lmax) {
      rc = fail(msg, msg_len, "instr %d: bad layer %d", i, r->layer);
      goto out;
    }
    if (r->sig_ctr >= (uint32_t)n_ctr) {
      rc = fail(msg, msg_len, "instr %d: bad signal counter", i);
      goto out;
    }
    int first_qkv = r->op == OQKV && r->layer == 0;
    if (first_qkv != (r->wait_ctr == NONE)) {
      rc = fail(msg, msg_len, "instr %d: only layer-0 QKV may start without a wait", i);
      goto out;
    }
    if (r->wait_ctr != NONE && r->wait_ctr >= (uint32_t)n_ctr) {
      rc = fail(msg, msg_len, "instr %d: bad wait counter", i);
      goto out;
    }
    push(&BYOP(r->op, r->op == OLM ? 0 : r->layer), i);
    push(&c.events[r->sig_ctr], i);
    if (r->op == OQKV) {
      if (r->g < 0 || r->g >= nkv || r->nrows == 0 ||
          r->row0 < (uint32_t)(r->g * GROUP_ROWS) ||
          r->row0 + r->nrows > (uint32_t)((r->g + 1) * GROUP_ROWS)) {
        rc = fail(msg, msg_len, "instr %d: QKV rows outside group %d", i, r->g);
        goto out;
      }
      push(&qkv_g[r->layer * nkv + r->g], i);
    }
    if (r->op == OATTN) {
      if (r->b < 0 || r->b >= B || r->g < 0 || r->g >= nkv || r->nchunk == 0 ||
          r->chunk >= r->nchunk || r->sig2_ctr >= (uint32_t)n_ctr ||
          r->sig2_after != r->nchunk) {
        rc = fail(msg, msg_len, "instr %d: bad attention fields", i);
        goto out;
      }
      int m = merge_id(s, r->layer, r->b, r->g);
      if (c.chunks[m].n == 0) nchunk_of[m] = r->nchunk;
      if (nchunk_of[m] != r->nchunk) {
        rc = fail(msg, msg_len, "instr %d: chunk count differs within its group", i);
        goto out;
      }
      push(&c.chunks[m], i);
    } else if (r->sig2_ctr != NONE) {
      if (r->nchunk == 0 || r->chunk >= r->nchunk || r->sig2_ctr >= (uint32_t)n_ctr ||
          r->sig2_after != r->nchunk) {
        rc = fail(msg, msg_len, "instr %d: bad split-projection fields", i);
        goto out;
      }
      const uint64_t key = ((uint64_t)r->op << 56) | ((uint64_t)(uint32_t)r->layer << 32) | r->row0;
      size_t h = (size_t)((key * 0x9E3779B97F4A7C15ULL) >> 20) % hcap;
      while (hkey[h] && hkey[h] != key + 1) h = (h + 1) % hcap;
      if (!hkey[h]) {
        hkey[h] = key + 1;
        hval[h] = n_split++;
      }
      int m = M_att + hval[h];
      if (c.chunks[m].n == 0) nchunk_of[m] = r->nchunk;
      if (nchunk_of[m] != r->nchunk || c.r[c.chunks[m].n ? c.chunks[m].v[0] : i].nrows != r->nrows) {
        rc = fail(msg, msg_len, "instr %d: slices of one row block disagree", i);
        goto out;
      }
      push(&c.chunks[m], i);
    }
  }
  /* merge nodes: one per (layer, sequence, group) of attention and one per
     split row block; they signal sig2 */
  for (int m = 0; m < M_att + n_split; ++m) {
    ilist *ch = &c.chunks[m];
    if ((uint32_t)ch->n != nchunk_of[m] || ch->n == 0) {
      rc = fail(msg, msg_len, "attention group %d has %d of %u chunks", m, ch->n, nchunk_of[m]);
      goto out;
    }
    if (m >= M_att) { /* slices must be 0..nchunk-1, each once */
      unsigned char *seen = (unsigned char *)calloc(nchunk_of[m], 1);
      int dup = 0;
      for (int j = 0; j < ch->n; ++j) dup |= seen[c.r[ch->v[j]].chunk]++;
      free(seen);
      if (dup) {
        rc = fail(msg, msg_len, "split row block %d: a slice appears twice", m - M_att);
        goto out;
      }
    }
    uint32_t sig2 = c.r[ch->v[0]].sig2_ctr, arr = c.r[ch->v[0]].sig_ctr;
    for (int j = 0; j < ch->n; ++j)
      if (c.r[ch->v[j]].sig2_ctr != sig2 || c.r[ch->v[j]].sig_ctr != arr) {
        rc = fail(msg, msg_len, "attention group %d: chunks disagree on counters", m);
        goto out;
      }
    if ((uint32_t)c.events[arr].n != nchunk_of[m]) {
      rc = fail(msg, msg_len, "attention group %d: arrival counter shared with other work", m);
      goto out;
    }
    push(&c.events[sig2], N + m);
  }

  /* 2. coverage: every output element of every op written exactly once */
  cov_qkv = (unsigned char *)calloc((size_t)L * QKV_ROWS, 1);
  cov_h = (unsigned char *)calloc((size_t)L * s->F, 1);
  cov_x3 = (unsigned char *)calloc((size_t)L * s->H, 1);
  cov_x5 = (unsigned char *)calloc((size_t)L * s->H, 1);
  cov_lm = (unsigned char *)calloc((size_t)s->V, 1);
  cov_att = (unsigned char *)calloc((size_t)M_att * 4096, 1);
  for (int i = 0; i < N; ++i) {
    rec_t *r = &c.r[i];
    unsigned char *cov = 0;
    uint32_t lim = 0;
    switch (r->op) {
      case OQKV: cov = cov_qkv + (size_t)r->layer * QKV_ROWS; lim = QKV_ROWS; break;
      case OGATEUP: cov = cov_h + (size_t)r->layer * s->F; lim = s->F; break;
      case OOPROJ: cov = cov_x3 + (size_t)r->layer * s->H; lim = s->H; break;
      case ODOWN: cov = cov_x5 + (size_t)r->layer * s->H; lim = s->H; break;
      case OLM: cov = cov_lm; lim = s->V; break;
      case OATTN: {
        if (r->nchunk > 4096) {
          rc = fail(msg, msg_len, "instr %d: too many chunks", i);
          goto out;
        }
        unsigned char *a = cov_att + (size_t)merge_id(s, r->layer, r->b, r->g) * 4096;
        if (a[r->chunk]++) {
          rc = fail(msg, msg_len, "instr %d: attention chunk written twice", i);
          goto out;
        }
        continue;
      }
    }
    if (r->sig2_ctr != NONE && r->chunk != 0) continue; /* a split block covers its rows once */
    if (r->nrows == 0 || r->row0 + r->nrows > lim) {
      rc = fail(msg, msg_len, "instr %d: rows [%u,%u) outside [0,%u)", i, r->row0,
                r->row0 + r->nrows, lim);
      goto out;
    }
    for (uint32_t k = r->row0; k < r->row0 + r->nrows; ++k)
      if (cov[k]++) {
        rc = fail(msg, msg_len, "instr %d: output row %u written twice", i, k);
        goto out;
      }
  }
  {
    size_t sizes[5] = {(size_t)L * QKV_ROWS, (size_t)L * s->F, (size_t)L * s->H,
                       (size_t)L * s->H, (size_t)s->V};
    unsigned char *covs[5] = {cov_qkv, cov_h, cov_x3, cov_x5, cov_lm};
    const char *names[5] = {"qkv", "gate/up", "o-proj", "down", "lm-head"};
    for (int t = 0; t < 5; ++t)
      for (size_t k = 0; k < sizes[t]; ++k)
        if (covs[t][k] != 1) {
          rc = fail(msg, msg_len, "%s output element %zu not written", names[t], k);
          goto out;
        }
  }

  /* 3. wait targets and queue order */
  for (int i = 0; i < N; ++i) {
    rec_t *r = &c.r[i];
    if (r->wait_ctr == NONE) continue;
    ilist *ev = &c.events[r->wait_ctr];
    if ((uint32_t)ev->n != r->wait_tgt) {
      rc = fail(msg, msg_len, "instr %d waits for %u signals but counter %u gets %d per step", i,
                r->wait_tgt, r->wait_ctr, ev->n);
      goto out;
    }
    for (int j = 0; j < ev->n; ++j) {
      int x = ev->v[j];
      int last = x;
      if (x >= N) {
        ilist *ch = &c.chunks[x - N];
        last = 0;
        for (int k = 0; k < ch->n; ++k)
          if (ch->v[k] > last) last = ch->v[k];
      }
      if (last >= i) {
        rc = fail(msg, msg_len, "instr %d waits on work queued at or after it (%d)", i, last);
        goto out;
      }
    }
  }
  for (int k = 0; k < n_ctr; ++k) inc_out[k] = (uint32_t)c.events[k].n;

  /* 4. data-flow hazards: every producer (read-after-write) and every earlier
        reader of overwritten data (write-after-read) must be complete before
        an instruction starts, through the chain of counters it waits on. */
  for (int i = 0; i < N && rc == 0; ++i) {
    rec_t *r = &c.r[i];
    const int l = r->layer;
    const uint64_t *cl = r->wait_ctr == NONE ? 0 : closure_of_ctr(&c, r->wait_ctr);
    if (c.cycle) {
      rc = fail(msg, msg_len, "counter dependency cycle");
      break;
    }
#define NEED_LIST(lst, what)                                                          \
  for (int j = 0; j < (lst).n; ++j)                                                   \
    if (!cl || !has(cl, (lst).v[j])) {                                                \
      rc = fail(msg, msg_len, "instr %d (op %d layer %d) may start before %s %d", i, \
                r->op, l, what, (lst).v[j]);                                          \
      goto out;                                                                       \
    }
#define NEED_NODE(node, what)                                                         \
  if (!cl || !has(cl, (node))) {                                                      \
    rc = fail(msg, msg_len, "instr %d (op %d layer %d) may start before %s", i,      \
              r->op, l, what);                                                        \
    goto out;                                                                         \
  }
    switch (r->op) {
      case OQKV:
        if (l > 0) {
          NEED_LIST(BYOP(ODOWN, l - 1), "down tile");   /* x it normalises */
          for (int b = 0; b < B; ++b)                    /* q/k/v it overwrites */
            NEED_LIST(c.chunks[merge_id(s, l - 1, b, r->g)], "attention chunk");
        }
        break;
      case OATTN:
        NEED_LIST(qkv_g[l * nkv + r->g], "qkv tile"); /* q, k, v of its group */
        if (l > 0) {
          NEED_NODE(N + merge_id(s, l - 1, r->b, r->g), "previous merge of its group");
          NEED_LIST(BYOP(OOPROJ, l - 1), "o-proj tile"); /* attention rows it overwrites */
        }
        break;
      case OOPROJ:
        for (int m = 0; m < B * nkv; ++m) NEED_NODE(N + l * B * nkv + m, "attention merge");
        NEED_LIST(BYOP(OQKV, l), "qkv tile"); /* readers of the x rows it updates */
        if (l > 0) NEED_LIST(BYOP(ODOWN, l - 1), "down tile");
        break;
      case OGATEUP:
        NEED_LIST(BYOP(OOPROJ, l), "o-proj tile");
        if (l > 0) NEED_LIST(BYOP(ODOWN, l - 1), "down tile (reader of h)");
        break;
      case ODOWN:
        NEED_LIST(BYOP(OGATEUP, l), "gate/up tile");
        NEED_LIST(BYOP(OOPROJ, l), "o-proj tile");
        break;
      case OLM:
        NEED_LIST(BYOP(ODOWN, L - 1), "down tile");
        break;
    }
  }

  /* 5. static per-SM lists: a partition of the queue, each list in queue order */
  if (list_off && list_idx && rc == 0) {
    unsigned char *seen = (unsigned char *)calloc((size_t)N, 1);
    if (list_off[0] != 0 || list_off[S] != (uint32_t)N) rc = fail(msg, msg_len, "lists do not cover the queue");
    for (int sm = 0; sm < S && rc == 0; ++sm)
      for (uint32_t k = list_off[sm]; k < list_off[sm + 1] && rc == 0; ++k) {
        uint32_t x = list_idx[k];
        if (x >= (uint32_t)N || seen[x]++) rc = fail(msg, msg_len, "list entry %u repeated or out of range", x);
        else if (k > list_off[sm] && list_idx[k - 1] >= x) rc = fail(msg, msg_len, "list of SM %d not in queue order", sm);
      }
    free(seen);
  }
#undef NEED_LIST
#undef NEED_NODE
#undef BYOP
out:
  if (c.clo)
    for (int k = 0; k < n_ctr; ++k) free(c.clo[k]);
  free(c.clo);
  free(c.state);
  free(c.r);
  free_lists(c.events, n_ctr);
  free_lists(c.chunks, c.M);
  free_lists(byop, 7 * (L + 1));
  free_lists(qkv_g, L * nkv);
  free(nchunk_of);
  free(hkey);
  free(hval);
  free(cov_qkv);
  free(cov_h);
  free(cov_x3);
  free(cov_x5);
  free(cov_lm);
  free(cov_att);
  return rc;
}

/* ---- deadlock search ------------------------------------------------------
 * Virtual SMs each hold a FIFO of claimed instructions (depth fifo_depth) and
 * finish them in claim order; an instruction can finish once its counter has
 * reached its target.  Dynamic mode claims the next queue entry; static mode
 * takes the next entry of the SM's own list.  Hybrid lists (att_first not
 * NULL) hold, in place of layer l's attention instructions, one entry with
 * bit 31 set and l below it: there the SM claims att_first[l] + q[l]++ from
 * that layer's queue until all att_count are claimed, then goes on with its
 * list.  Every step picks one enabled action at random (seeded); finding no
 * enabled action with work left is a deadlock. */
static uint64_t rng_next(uint64_t *s) {
  uint64_t z = (*s += 0x9E3779B97F4A7C15ULL);
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ULL;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBULL;
  return z ^ (z >> 31);
}

static void apply_done(const rec_t *r, uint32_t *cnt) {
  cnt[r->sig_ctr] += 1;
  if (r->sig2_ctr != NONE && cnt[r->sig_ctr] == r->sig2_after) cnt[r->sig2_ctr] += 1;
}

static int ready(const rec_t *r, const uint32_t *cnt) {
  return r->wait_ctr == NONE || cnt[r->wait_ctr] >= r->wait_tgt;
}

#define ATT_MARK 0x80000000u

int or_simulate(const void *table, int N, int n_ctr, int S, int D, uint64_t seed, int trials,
                const uint32_t *list_off, const uint32_t *list_idx, const uint32_t *att_first,
                int n_att, int att_count, char *msg, int msg_len) {
  if (S <= 0 || D <= 0 || N <= 0) return fail(msg, msg_len, "bad arguments");
  rec_t *r = (rec_t *)malloc(sizeof(rec_t) * (size_t)N);
  for (int i = 0; i < N; ++i) decode(table, i, &r[i]);
  uint32_t *cnt = (uint32_t *)malloc(sizeof(uint32_t) * (size_t)n_ctr);
  int *fifo = (int *)malloc(sizeof(int) * (size_t)S * D);
  int *fh = (int *)malloc(sizeof(int) * (size_t)S), *fl = (int *)malloc(sizeof(int) * (size_t)S);
  uint32_t *lp = (uint32_t *)malloc(sizeof(uint32_t) * (size_t)S);
  int *acts = (int *)malloc(sizeof(int) * (size_t)2 * S);
  int *att_l = (int *)malloc(sizeof(int) * (size_t)S);       /* hybrid: layer being claimed */
  int *aq = (int *)calloc((size_t)(n_att > 0 ? n_att : 1), sizeof(int));
  unsigned char *seen = (unsigned char *)malloc((size_t)N);
  int rc = 0;
  for (int t = 0; t < trials && rc == 0; ++t) {
    uint64_t st = seed * 1000003ULL + (uint64_t)t;
    memset(cnt, 0, sizeof(uint32_t) * (size_t)n_ctr);
    for (int s = 0; s < S; ++s) {
      fh[s] = fl[s] = 0;
      lp[s] = list_off ? list_off[s] : 0;
      att_l[s] = -1;
    }
    for (int l = 0; l < n_att; ++l) aq[l] = 0;
    memset(seen, 0, (size_t)N);
    int nx = 0, done = 0;
    while (done < N) {
      int na = 0;
      for (int s = 0; s < S; ++s) {
        /* hybrid: step over exhausted queues and onto markers until a claim
           is possible or the list ends (no instruction is taken here) */
        while (att_first && list_off) {
          if (att_l[s] >= 0 && aq[att_l[s]] < att_count) break;
          att_l[s] = -1;
          if (lp[s] >= list_off[s + 1] || !(list_idx[lp[s]] & ATT_MARK)) break;
          const uint32_t l = list_idx[lp[s]++] & ~ATT_MARK;
          if ((int)l >= n_att) {
            rc = fail(msg, msg_len, "list marker for layer %u of %d", l, n_att);
            break;
          }
          att_l[s] = (int)l;
        }
        if (rc) break;
        int can_claim = fl[s] < D && (att_l[s] >= 0 || (list_off ? lp[s] < list_off[s + 1] : nx < N));
        if (can_claim) acts[na++] = 2 * s;
        if (fl[s] > 0 && ready(&r[fifo[s * D + fh[s]]], cnt)) acts[na++] = 2 * s + 1;
      }
      if (rc) break;
      if (na == 0) {
        rc = fail(msg, msg_len, "deadlock in trial %d with %d of %d done", t, done, N);
        break;
      }
      int a = acts[rng_next(&st) % (uint64_t)na], s = a >> 1;
      if (a & 1) {
        int x = fifo[s * D + fh[s]];
        fh[s] = (fh[s] + 1) % D;
        fl[s]--;
        apply_done(&r[x], cnt);
        done++;
      } else {
        int x;
        if (att_l[s] >= 0) x = (int)att_first[att_l[s]] + aq[att_l[s]]++;
        else x = list_off ? (int)list_idx[lp[s]++] : nx++;
        if (x < 0 || x >= N || seen[x]++) {
          rc = fail(msg, msg_len, "instruction %d out of range or claimed twice", x);
          break;
        }
        fifo[s * D + (fh[s] + fl[s]) % D] = x;
        fl[s]++;
      }
    }
  }
  free(r);
  free(cnt);
  free(fifo);
  free(fh);
  free(fl);
  free(lp);
  free(acts);
  free(att_l);
  free(aq);
  free(seen);
  return rc;
}

/* Exhaustive search over every interleaving of two virtual SMs (dynamic
 * queue), for small tables.  A state is (next queue index, FIFO of SM 0,
 * FIFO of SM 1); everything claimed and not in a FIFO is done.  Returns the
 * number of distinct states reached, -1 on a deadlock, -2 if max_states is
 * exceeded. */
typedef struct {
  int nx, l0, l1;
  int f0[8], f1[8];
} xstate;

static uint64_t xhash(const xstate *s) {
  uint64_t h = (uint64_t)s->nx * 1315423911ULL + (uint64_t)s->l0 * 31 + (uint64_t)s->l1 * 131;
  for (int i = 0; i < s->l0; ++i) h = rng_next(&h) ^ (uint64_t)s->f0[i];
  h ^= 0xABCDEFULL;
  for (int i = 0; i < s->l1; ++i) h = rng_next(&h) ^ (uint64_t)s->f1[i];
  return h;
}
static int xeq(const xstate *a, const xstate *b) {
  if (a->nx != b->nx || a->l0 != b->l0 || a->l1 != b->l1) return 0;
  for (int i = 0; i < a->l0; ++i)
    if (a->f0[i] != b->f0[i]) return 0;
  for (int i = 0; i < a->l1; ++i)
    if (a->f1[i] != b->f1[i]) return 0;
  return 1;
}

long or_explore(const void *table, int N, int n_ctr, int D, long max_states, char *msg,
                int msg_len) {
  if (D < 1 || D > 8 || N <= 0 || max_states <= 0) return fail(msg, msg_len, "bad arguments");
  rec_t *r = (rec_t *)malloc(sizeof(rec_t) * (size_t)N);
  for (int i = 0; i < N; ++i) decode(table, i, &r[i]);
  long cap = 1;
  while (cap < 2 * max_states) cap <<= 1;
  xstate *tab = (xstate *)malloc(sizeof(xstate) * (size_t)cap);
  unsigned char *used = (unsigned char *)calloc((size_t)cap, 1);
  xstate *stack = (xstate *)malloc(sizeof(xstate) * (size_t)max_states);
  uint32_t *cnt = (uint32_t *)malloc(sizeof(uint32_t) * (size_t)n_ctr);
  unsigned char *pend = (unsigned char *)calloc((size_t)N, 1);
  long nstates = 0, sp = 0;
  long rc = 0;
  xstate s0;
  memset(&s0, 0, sizeof s0);
  stack[sp++] = s0;
  {
    uint64_t h = xhash(&s0) & (uint64_t)(cap - 1);
    used[h] = 1;
    tab[h] = s0;
    nstates = 1;
  }
  while (sp > 0) {
    xstate s = stack[--sp];
    /* counters of this state: every claimed instruction not pending is done */
    memset(cnt, 0, sizeof(uint32_t) * (size_t)n_ctr);
    for (int i = 0; i < s.l0; ++i) pend[s.f0[i]] = 1;
    for (int i = 0; i < s.l1; ++i) pend[s.f1[i]] = 1;
    for (int i = 0; i < s.nx; ++i)
      if (!pend[i]) apply_done(&r[i], cnt);
    for (int i = 0; i < s.l0; ++i) pend[s.f0[i]] = 0;
    for (int i = 0; i < s.l1; ++i) pend[s.f1[i]] = 0;
    xstate nxt[4];
    int nn = 0;
    if (s.l0 < D && s.nx < N) {
      nxt[nn] = s;
      nxt[nn].f0[nxt[nn].l0++] = s.nx;
      nxt[nn++].nx++;
    }
    if (s.l1 < D && s.nx < N) {
      nxt[nn] = s;
      nxt[nn].f1[nxt[nn].l1++] = s.nx;
      nxt[nn++].nx++;
    }
    if (s.l0 > 0 && ready(&r[s.f0[0]], cnt)) {
      nxt[nn] = s;
      memmove(nxt[nn].f0, nxt[nn].f0 + 1, sizeof(int) * 7);
      nxt[nn++].l0--;
    }
    if (s.l1 > 0 && ready(&r[s.f1[0]], cnt)) {
      nxt[nn] = s;
      memmove(nxt[nn].f1, nxt[nn].f1 + 1, sizeof(int) * 7);
      nxt[nn++].l1--;
    }
    int finished = s.nx == N && s.l0 == 0 && s.l1 == 0;
    if (nn == 0 && !finished) {
      rc = fail(msg, msg_len, "deadlock at queue index %d", s.nx);
      break;
    }
    for (int k = 0; k < nn; ++k) {
      uint64_t h = xhash(&nxt[k]) & (uint64_t)(cap - 1);
      int dup = 0;
      while (used[h]) {
        if (xeq(&tab[h], &nxt[k])) {
          dup = 1;
          break;
        }
        h = (h + 1) & (uint64_t)(cap - 1);
      }
      if (dup) continue;
      if (nstates >= max_states) {
        rc = -2;
        fail(msg, msg_len, "more than %ld states", max_states);
        goto done;
      }
      used[h] = 1;
      tab[h] = nxt[k];
      nstates++;
      stack[sp++] = nxt[k];
    }
  }
done:
  free(r);
  free(tab);
  free(used);
  free(stack);
  free(cnt);
  free(pend);
  return rc < 0 ? rc : nstates;
}

/* ---- run-time re-deal of batched attention slots ---------------------------
 * In batched plans run from static per-SM lists, whether an attention chunk
 * has keys to read depends on its sequence's position, known only when the
 * step runs.  So the slots of each layer's attention phase are re-dealt at
 * run time: the phase's instructions are listed with every chunk that has
 * work first and every empty chunk after, each part in queue order, and the
 * list slot holding the phase's j-th instruction executes the j-th of that
 * listing instead.  A chunk c of sequence b covers positions
 * [c * chunk, min((c + 1) * chunk, pos_b + 1)); it has work when that range
 * is not empty.
 *
 * Checked here, from the table alone:
 *  - each attention phase (a run of attention records of one layer) lists
 *    chunk-major, then sequence, then group, every (chunk, sequence, group)
 *    once;
 *  - the records of a phase differ only in chunk, sequence, group, their
 *    signal counter (one arrival counter per (sequence, group), consecutive
 *    in group, then sequence) and their wait counter (one per group,
 *    consecutive), so rewriting those fields of one record by the slot's
 *    offsets gives exactly the record of the instruction it is re-dealt to;
 *  - the executed lists are a partition of the queue in which every entry
 *    stays in its own phase.
 * Writes the executed index of every list slot to exec_idx (n_list entries;
 * list_idx may be NULL for the queue order itself, n_list = n_instr). */
int or_redeal(const void *table, int N, const or_shape *s, int attn_chunk,
              const int32_t *positions, const uint32_t *list_idx, int n_list,
              uint32_t *exec_idx, char *msg, int msg_len) {
  const int B = s->B, G = s->nkv;
  if (N <= 0 || B <= 0 || G <= 0 || attn_chunk <= 0 || n_list != N)
    return fail(msg, msg_len, "bad arguments");
  rec_t *r = (rec_t *)malloc(sizeof(rec_t) * (size_t)N);
  int *target = (int *)malloc(sizeof(int) * (size_t)N);  /* queue index -> executed index */
  int *order = (int *)malloc(sizeof(int) * (size_t)N);
  unsigned char *seen = (unsigned char *)calloc((size_t)N, 1);
  int rc = 0;
  for (int i = 0; i < N; ++i) {
    decode(table, i, &r[i]);
    target[i] = i;
  }
  for (int a = 0; a < N && rc == 0;) {
    if (r[a].op != OATTN) {
      ++a;
      continue;
    }
    int e = a;
    while (e < N && r[e].op == OATTN && r[e].layer == r[a].layer) ++e;
    const int n = e - a, C = (int)r[a].nchunk;
    if (C <= 0 || n != C * B * G) {
      rc = fail(msg, msg_len, "attention phase at %d: %d records for %d chunks x %d x %d", a, n,
                C, B, G);
      break;
    }
    for (int j = 0; j < n && rc == 0; ++j) {
      const rec_t *x = &r[a + j], *f = &r[a];
      const int c = j / (B * G), b = (j / G) % B, g = j % G;
      if ((int)x->chunk != c || x->b != b || x->g != g)
        rc = fail(msg, msg_len, "attention record %d is not chunk-major", a + j);
      else if (x->flags != f->flags || x->wait_tgt != f->wait_tgt || x->sig2_ctr != f->sig2_ctr ||
               x->sig2_after != f->sig2_after || x->row0 != f->row0 || x->nrows != f->nrows ||
               x->nchunk != f->nchunk)
        rc = fail(msg, msg_len, "attention record %d differs from its phase in a fixed field",
                  a + j);
      else if (x->sig_ctr != f->sig_ctr + (uint32_t)(b * G + g))
        rc = fail(msg, msg_len, "attention record %d: arrival counter not per (sequence, group)",
                  a + j);
      else if (x->wait_ctr != f->wait_ctr + (uint32_t)g)
        rc = fail(msg, msg_len, "attention record %d: wait counter not per group", a + j);
    }
    if (rc) break;
    /* the listing: chunks with work, then empty chunks, each in queue order */
    int k = 0;
    for (int pass = 0; pass < 2; ++pass)
      for (int j = 0; j < n; ++j) {
        const int c = j / (B * G), b = (j / G) % B;
        const long first = (long)c * attn_chunk;
        const long end_ = (long)positions[b] + 1 < first + attn_chunk ? (long)positions[b] + 1
                                                                       : first + attn_chunk;
        const int has_work = end_ > first;
        if (has_work == (pass == 0)) order[k++] = a + j;
      }
    for (int j = 0; j < n; ++j) target[a + j] = order[j];
    a = e;
  }
  for (int k = 0; k < n_list && rc == 0; ++k) {
    const uint32_t q = list_idx ? list_idx[k] : (uint32_t)k;
    if (q >= (uint32_t)N) {
      rc = fail(msg, msg_len, "list entry %u out of range", q);
      break;
    }
    const int x = target[q];
    if (seen[x]++) rc = fail(msg, msg_len, "instruction %d executed twice", x);
    else if (r[x].op != r[q].op || r[x].layer != r[q].layer)
      rc = fail(msg, msg_len, "slot of instruction %u moved out of its phase", q);
    exec_idx[k] = (uint32_t)x;
  }
  free(r);
  free(target);
  free(order);
  free(seen);
  return rc;
}
