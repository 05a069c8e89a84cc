/*
 * umm_oracle.c -- plain, slow CPU oracle of the EP<->TP reshard data plane.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product library links, includes
 * or calls this file; only the tests, the smoke check and the CPU-baseline leg
 * of the benchmark load it (through oracle/__init__.py).  It shares no header,
 * constant or helper with the CUDA path: every offset and index map below is
 * restated here from the method's description.
 *
 * Source: "Moebius: Serving Mixture-of-Expert Models with Seamless Runtime
 * Parallelism Switch" (paper review page):
 *   §3   "one model, two layouts": the bytes are identical, only ownership moves;
 *   §3.1 weight shapes  EP: W13 (E/P, 2I, H), W2 (E/P, H, I)
 *                       TP: W13 (E, 2I/P, H), W2 (E, H, I/P);
 *   §3.2 KV: EP keeps all heads of its own requests, TP keeps a head shard of
 *        every request, heads replicated over rank groups when KV heads < P
 *        (4 heads at TP-8 -> 2 ranks per head); paged KV moved through the
 *        page tables; TP->EP placement = sort by length descending, each
 *        request to the least-loaded rank;
 *   §4.2, Fig. 7: one unified buffer per rank, N+1 weight slots, TP layer i in
 *        slot i, EP layer i in slot i+1; EP->TP runs layers ascending, TP->EP
 *        descending;
 *   §4.3, Table 1: one read and one write per moved element.
 *
 * Readings of points the page leaves open (each is restated where it is used):
 *   R-1 buffer layout: region r = [weight slot 0..N][KV slot 0..N][attention
 *       slot 0..N] (attention slots only when there are attention weights,
 *       R-16); KV and attention use the same N+1 slot mapping as the weights;
 *       the P regions are followed by a workspace.  Alignments: W2 at 256 B inside a slot, slot strides at
 *       4 KiB, region stride at 2 MiB.  K half then V half in a KV slot, each
 *       half sized for the TP view.
 *   R-2 TP rank q's 2I/P rows of W13 = gate rows [q*Ip,(q+1)*Ip) followed by
 *       up rows [q*Ip,(q+1)*Ip) (split 0), or rows [q*2Ip,(q+1)*2Ip) (split 1).
 *   R-3 Hkv >= P: rank q holds heads [q*Hkv/P, (q+1)*Hkv/P);
 *       Hkv <  P: rank q holds head floor(q*Hkv/P).
 *   R-4 TP->EP reads each head from the lowest rank that holds it.
 *   R-5 placement load = tokens; order (len desc, list key asc); load ties go
 *       to the lowest rank.
 *   R-6 local order inside an EP rank = ascending list key.
 *   R-7 pages are handed out in list order from a caller-given free list.
 *   R-8 bytes that are not a destination keep their previous contents.
 *   R-16 attention weights (§3.1, memory-saving variant: only the active
 *       layout is kept; TP->EP rebuilds it with an all-gather).  EP (DP
 *       attention): every rank holds the full Wqkv = [Hq query heads][Hkv key
 *       heads][Hkv value heads], each head Dh rows of H, and Wo [H][Hq*Dh].
 *       TP: rank q holds query heads [q*Hq/P, (q+1)*Hq/P), its KV heads (R-3)
 *       for K then V, and the Wo columns of its query heads.  Both views use
 *       the same offsets inside an attention slot (Wqkv at 0, Wo at a
 *       256-byte boundary after the full Wqkv); N+1 slots as for the weights.
 *
 * All data is moved as raw bytes (bf16 = 2 opaque bytes); nothing passes
 * through floating point.
 */
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* ---- dims / layout vectors exchanged with the Python wrapper (int64) ---- */
enum {
  OD_P, OD_E, OD_H, OD_I, OD_N, OD_HKV, OD_HD, OD_PS, OD_PAGES_TP,
  OD_MAX_REQ, OD_MAX_PAGES, OD_W13_SPLIT, OD_HQ, OD_COUNT
};
enum {
  OL_REGION_STRIDE, OL_WSLOT_STRIDE, OL_W13_OFF, OL_W2_OFF, OL_KVSLOT_STRIDE,
  OL_KV_V_OFF, OL_KVSLOTS_OFF, OL_WS_OFF, OL_PAGES_EP, OL_PAGES_TP, OL_H_TP,
  OL_ATTN_STRIDE, OL_ATTN_WO_OFF, OL_ATTNSLOTS_OFF, OL_COUNT
};

/* error flags the oracle expects a KV/assign call to raise (bit values) */
#define ORC_F_BAD_REQUEST 1u
#define ORC_F_CAPACITY    2u
#define ORC_F_PAGE_OOB    4u
#define ORC_F_DUP_PAGE    8u

static int g_threads = 1;
void orc_set_threads(int n) { g_threads = n < 1 ? 1 : n; }
int orc_max_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}

static int64_t round_up(int64_t x, int64_t a) { return (x + a - 1) / a * a; }

/* R-1: offsets of every part of the unified buffer. */
void orc_layout(const int64_t *d, int64_t *L) {
  int64_t P = d[OD_P], E = d[OD_E], H = d[OD_H], I = d[OD_I], N = d[OD_N];
  int64_t Hkv = d[OD_HKV], D = d[OD_HD], ps = d[OD_PS], pages_tp = d[OD_PAGES_TP];
  int64_t El = E / P;
  int64_t w13 = El * 2 * I * H * 2;          /* bytes of W13 in one region slot */
  int64_t w2 = El * H * I * 2;               /* bytes of W2 in one region slot  */
  int64_t w2_off = round_up(w13, 256);
  int64_t wslot = (E > 0) ? round_up(w2_off + w2, 4096) : 0;
  int64_t h_tp = (Hkv >= P) ? Hkv / P : 1;
  int64_t half = (Hkv > 0) ? pages_tp * ps * h_tp * D * 2 : 0;
  int64_t v_off = round_up(half, 256);
  int64_t kvslot = (Hkv > 0) ? round_up(v_off + half, 4096) : 0;
  int64_t Hq = d[OD_HQ];
  int64_t qkv = (Hq > 0) ? (Hq + 2 * Hkv) * D * H * 2 : 0;     /* full Wqkv bytes */
  int64_t wo_off = round_up(qkv, 256);
  int64_t attnslot = (Hq > 0) ? round_up(wo_off + H * Hq * D * 2, 4096) : 0;
  int64_t region = round_up((N + 1) * (wslot + kvslot + attnslot), (int64_t)2 << 20);
  memset(L, 0, sizeof(int64_t) * OL_COUNT);
  L[OL_REGION_STRIDE] = region;
  L[OL_WSLOT_STRIDE] = wslot;
  L[OL_W13_OFF] = 0;
  L[OL_W2_OFF] = w2_off;
  L[OL_KVSLOT_STRIDE] = kvslot;
  L[OL_KV_V_OFF] = v_off;
  L[OL_KVSLOTS_OFF] = (N + 1) * wslot;
  L[OL_WS_OFF] = P * region;
  L[OL_PAGES_EP] = (Hkv > 0) ? pages_tp * h_tp / Hkv : 0;
  L[OL_PAGES_TP] = pages_tp;
  L[OL_H_TP] = (Hkv > 0) ? h_tp : 0;
  L[OL_ATTN_STRIDE] = attnslot;
  L[OL_ATTN_WO_OFF] = wo_off;
  L[OL_ATTNSLOTS_OFF] = (N + 1) * (wslot + kvslot);
}

/* byte offset of weight slot s of region r */
static int64_t wslot_at(const int64_t *L, int64_t r, int64_t s) {
  return r * L[OL_REGION_STRIDE] + s * L[OL_WSLOT_STRIDE];
}
/* byte offset of KV slot s of region r, half c (0 = K, 1 = V) */
static int64_t kvslot_at(const int64_t *L, int64_t r, int64_t s, int64_t c) {
  return r * L[OL_REGION_STRIDE] + L[OL_KVSLOTS_OFF] + s * L[OL_KVSLOT_STRIDE] + c * L[OL_KV_V_OFF];
}

static void copy2(const uint8_t *src, uint8_t *dst, int64_t from, int64_t to) {
  dst[to] = src[from];
  dst[to + 1] = src[from + 1];
}

/* ------------------------------------------------------------------------ */
/* Weights                                                                   */
/* ------------------------------------------------------------------------ */

/* §3.1: the EP row j of expert (r, el) that becomes TP row `row` of expert e on
 * rank q.  R-2 decides which rows those are. */
static int64_t ep_row_of_tp_row(int64_t split, int64_t I, int64_t Ip, int64_t q, int64_t row) {
  if (split == 0) {
    int64_t g = row / Ip;          /* 0 = gate (W1), 1 = up (W3) */
    int64_t ii = row % Ip;
    return g * I + q * Ip + ii;
  }
  return q * 2 * Ip + row;
}

/* One weight layer EP -> TP: every TP element of slot `tp_slot` is assigned
 * the EP element of slot `ep_slot` that holds the same logical value.
 * Reads `src`, writes `dst` (the same buffer for in-place use). */
static void weights_layer_ep2tp(const uint8_t *src, uint8_t *dst, const int64_t *d,
                                const int64_t *L, int64_t ep_slot, int64_t tp_slot) {
  int64_t P = d[OD_P], E = d[OD_E], H = d[OD_H], I = d[OD_I], split = d[OD_W13_SPLIT];
  int64_t El = E / P, Ip = I / P;
#pragma omp parallel for num_threads(g_threads) schedule(static) if (g_threads > 1)
  for (int64_t q = 0; q < P; ++q) {
    for (int64_t e = 0; e < E; ++e) {
      int64_t r = e / El, el = e % El;     /* EP owner of expert e */
      /* W13: TP (E, 2Ip, H) on rank q  <-  EP (El, 2I, H) on rank r */
      for (int64_t row = 0; row < 2 * Ip; ++row) {
        int64_t j = ep_row_of_tp_row(split, I, Ip, q, row);
        for (int64_t h = 0; h < H; ++h) {
          int64_t from = wslot_at(L, r, ep_slot) + L[OL_W13_OFF] + ((el * 2 * I + j) * H + h) * 2;
          int64_t to = wslot_at(L, q, tp_slot) + L[OL_W13_OFF] + ((e * 2 * Ip + row) * H + h) * 2;
          copy2(src, dst, from, to);
        }
      }
      /* W2: TP (E, H, Ip) on rank q  <-  EP (El, H, I) on rank r, columns q*Ip.. */
      for (int64_t h = 0; h < H; ++h) {
        for (int64_t c = 0; c < Ip; ++c) {
          int64_t i = q * Ip + c;
          int64_t from = wslot_at(L, r, ep_slot) + L[OL_W2_OFF] + ((el * H + h) * I + i) * 2;
          int64_t to = wslot_at(L, q, tp_slot) + L[OL_W2_OFF] + ((e * H + h) * Ip + c) * 2;
          copy2(src, dst, from, to);
        }
      }
    }
  }
}

/* One weight layer TP -> EP, written from the EP side: every EP element finds
 * the TP rank and row that hold it (the inverse of the map above, derived
 * separately so that a round trip checks the two against each other). */
static void weights_layer_tp2ep(const uint8_t *src, uint8_t *dst, const int64_t *d,
                                const int64_t *L, int64_t tp_slot, int64_t ep_slot) {
  int64_t P = d[OD_P], E = d[OD_E], H = d[OD_H], I = d[OD_I], split = d[OD_W13_SPLIT];
  int64_t El = E / P, Ip = I / P;
#pragma omp parallel for num_threads(g_threads) schedule(static) if (g_threads > 1)
  for (int64_t r = 0; r < P; ++r) {
    for (int64_t el = 0; el < El; ++el) {
      int64_t e = r * El + el;
      for (int64_t j = 0; j < 2 * I; ++j) {
        int64_t q, row;
        if (split == 0) {
          int64_t g = j / I, i = j % I;      /* gate or up, intermediate index */
          q = i / Ip;
          row = g * Ip + i % Ip;
        } else {
          q = j / (2 * Ip);
          row = j % (2 * Ip);
        }
        for (int64_t h = 0; h < H; ++h) {
          int64_t from = wslot_at(L, q, tp_slot) + L[OL_W13_OFF] + ((e * 2 * Ip + row) * H + h) * 2;
          int64_t to = wslot_at(L, r, ep_slot) + L[OL_W13_OFF] + ((el * 2 * I + j) * H + h) * 2;
          copy2(src, dst, from, to);
        }
      }
      for (int64_t h = 0; h < H; ++h) {
        for (int64_t i = 0; i < I; ++i) {
          int64_t q = i / Ip, c = i % Ip;
          int64_t from = wslot_at(L, q, tp_slot) + L[OL_W2_OFF] + ((e * H + h) * Ip + c) * 2;
          int64_t to = wslot_at(L, r, ep_slot) + L[OL_W2_OFF] + ((el * H + h) * I + i) * 2;
          copy2(src, dst, from, to);
        }
      }
    }
  }
}

/* Whole EP -> TP weight switch (§4.2, Fig. 7): TP layer l lives in slot l, EP
 * layer l in slot l+1.  `order` = +1 walks layers ascending (the method's
 * order); -1 walks them descending (only used by a test that shows the
 * in-place result then goes wrong). */
void orc_weights_ep2tp(const uint8_t *src, uint8_t *dst, const int64_t *d, int order) {
  int64_t L[OL_COUNT];
  orc_layout(d, L);
  int64_t N = d[OD_N];
  for (int64_t t = 0; t < N; ++t) {
    int64_t l = (order >= 0) ? t : N - 1 - t;
    weights_layer_ep2tp(src, dst, d, L, l + 1, l);
  }
}

/* Whole TP -> EP weight switch: layers descending (order = -1 is the method's). */
void orc_weights_tp2ep(const uint8_t *src, uint8_t *dst, const int64_t *d, int order) {
  int64_t L[OL_COUNT];
  orc_layout(d, L);
  int64_t N = d[OD_N];
  for (int64_t t = 0; t < N; ++t) {
    int64_t l = (order < 0) ? N - 1 - t : t;
    weights_layer_tp2ep(src, dst, d, L, l, l + 1);
  }
}

/* Element maps for sampled checks at sizes the oracle cannot run whole.
 * TP W13 element (q, e, row, h) -> EP coordinates (r, el, j, h); returns the
 * byte offsets of the EP source (slot ep_slot) and TP destination (tp_slot). */
void orc_w13_tp_elem(const int64_t *d, int64_t q, int64_t e, int64_t row, int64_t h,
                     int64_t ep_slot, int64_t tp_slot, int64_t *src_off, int64_t *dst_off) {
  int64_t L[OL_COUNT];
  orc_layout(d, L);
  int64_t P = d[OD_P], E = d[OD_E], H = d[OD_H], I = d[OD_I];
  int64_t El = E / P, Ip = I / P;
  int64_t r = e / El, el = e % El;
  int64_t j = ep_row_of_tp_row(d[OD_W13_SPLIT], I, Ip, q, row);
  *src_off = wslot_at(L, r, ep_slot) + L[OL_W13_OFF] + ((el * 2 * I + j) * H + h) * 2;
  *dst_off = wslot_at(L, q, tp_slot) + L[OL_W13_OFF] + ((e * 2 * Ip + row) * H + h) * 2;
}

/* TP W2 element (q, e, h, c) -> EP source / TP destination byte offsets. */
void orc_w2_tp_elem(const int64_t *d, int64_t q, int64_t e, int64_t h, int64_t c,
                    int64_t ep_slot, int64_t tp_slot, int64_t *src_off, int64_t *dst_off) {
  int64_t L[OL_COUNT];
  orc_layout(d, L);
  int64_t P = d[OD_P], E = d[OD_E], H = d[OD_H], I = d[OD_I];
  int64_t El = E / P, Ip = I / P;
  int64_t r = e / El, el = e % El;
  *src_off = wslot_at(L, r, ep_slot) + L[OL_W2_OFF] + ((el * H + h) * I + q * Ip + c) * 2;
  *dst_off = wslot_at(L, q, tp_slot) + L[OL_W2_OFF] + ((e * H + h) * Ip + c) * 2;
}

/* ------------------------------------------------------------------------ */
/* KV cache                                                                  */
/* ------------------------------------------------------------------------ */

/* R-3: does TP rank q hold KV head h, and at which local head index? */
static int holds_head(int64_t P, int64_t Hkv, int64_t q, int64_t h, int64_t *local) {
  if (Hkv >= P) {
    int64_t per = Hkv / P;
    if (h >= q * per && h < (q + 1) * per) { *local = h - q * per; return 1; }
    return 0;
  }
  if (q * Hkv / P == h) { *local = 0; return 1; }
  return 0;
}

static int64_t npages_of(int64_t len, int64_t ps) { return (len + ps - 1) / ps; }

/* Validation a KV call must run before it moves any byte (§4.5 capacity check,
 * page tables of §3.2).  dir 0 = EP->TP (src pool = EP of owner, dst = TP),
 * dir 1 = TP->EP (src = TP, dst = EP of owner).  Returns a bit set of
 * ORC_F_* flags; 0 = the call may run. */
uint32_t orc_kv_validate(const int64_t *d, int dir, int64_t R, int64_t maxp,
                         const int32_t *lens, const int32_t *owner,
                         const int32_t *ep_pt, const int32_t *tp_pt) {
  int64_t L[OL_COUNT];
  orc_layout(d, L);
  int64_t P = d[OD_P], ps = d[OD_PS];
  int64_t pages_ep = L[OL_PAGES_EP], pages_tp = L[OL_PAGES_TP];
  uint32_t flags = 0;
  int64_t total = 0;
  int64_t *per_region = calloc((size_t)P, sizeof(int64_t));
  for (int64_t k = 0; k < R; ++k) {
    if (lens[k] < 0 || (int64_t)lens[k] > maxp * ps || owner[k] < 0 || owner[k] >= P) {
      flags |= ORC_F_BAD_REQUEST;
      continue;
    }
    int64_t np = npages_of(lens[k], ps);
    total += np;
    per_region[owner[k]] += np;
  }
  if (flags) { free(per_region); return flags; }
  if (total > d[OD_MAX_PAGES]) flags |= ORC_F_CAPACITY;
  if (dir == 0 && total > pages_tp) flags |= ORC_F_CAPACITY;
  if (dir == 1)
    for (int64_t r = 0; r < P; ++r)
      if (per_region[r] > pages_ep) flags |= ORC_F_CAPACITY;
  free(per_region);
  if (flags) return flags;
  /* page ids in range; destinations used at most once; and, since a page
   * holds the tokens of one request only (§3.2 page tables; no prefix sharing
   * in the setting of §6.1), the TP pages a TP->EP switch reads are distinct
   * too */
  int64_t dst_pool = (dir == 0) ? pages_tp : P * pages_ep;
  uint8_t *used = calloc((size_t)(dst_pool > 0 ? dst_pool : 1), 1);
  uint8_t *tp_used = calloc((size_t)(pages_tp > 0 ? pages_tp : 1), 1);
  for (int64_t k = 0; k < R; ++k) {
    int64_t np = npages_of(lens[k], ps);
    for (int64_t p = 0; p < np; ++p) {
      int64_t ep = ep_pt[k * maxp + p], tp = tp_pt[k * maxp + p];
      if (ep < 0 || ep >= pages_ep || tp < 0 || tp >= pages_tp) {
        flags |= ORC_F_PAGE_OOB;
        continue;
      }
      int64_t slot = (dir == 0) ? tp : owner[k] * pages_ep + ep;
      if (used[slot]) flags |= ORC_F_DUP_PAGE;
      used[slot] = 1;
      if (dir == 1) {
        if (tp_used[tp]) flags |= ORC_F_DUP_PAGE;
        tp_used[tp] = 1;
      }
    }
  }
  free(tp_used);
  free(used);
  return flags;
}

/* §3.2, Fig. 5: KV EP -> TP.  For every live token of every request, every K/V
 * half, every head and every TP rank holding that head, the head's D values
 * move from the owner's EP page to the rank's TP page.  Layers ascending,
 * EP layer l in KV slot l+1, TP layer l in KV slot l. */
uint32_t orc_kv_ep2tp(const uint8_t *src, uint8_t *dst, const int64_t *d, int64_t R, int64_t maxp,
                      const int32_t *lens, const int32_t *owner,
                      const int32_t *ep_pt, const int32_t *tp_pt, int order) {
  uint32_t flags = orc_kv_validate(d, 0, R, maxp, lens, owner, ep_pt, tp_pt);
  if (flags) return flags;
  int64_t L[OL_COUNT];
  orc_layout(d, L);
  int64_t P = d[OD_P], N = d[OD_N], Hkv = d[OD_HKV], D = d[OD_HD], ps = d[OD_PS];
  int64_t h_tp = L[OL_H_TP];
  for (int64_t t = 0; t < N; ++t) {
    int64_t l = (order >= 0) ? t : N - 1 - t;
#pragma omp parallel for num_threads(g_threads) schedule(dynamic, 1) if (g_threads > 1)
    for (int64_t k = 0; k < R; ++k) {
      int64_t o = owner[k];
      for (int64_t tok = 0; tok < lens[k]; ++tok) {
        int64_t p = tok / ps, s = tok % ps;
        int64_t sp = ep_pt[k * maxp + p], dp = tp_pt[k * maxp + p];
        for (int64_t c = 0; c < 2; ++c)
          for (int64_t h = 0; h < Hkv; ++h)
            for (int64_t q = 0; q < P; ++q) {
              int64_t hl;
              if (!holds_head(P, Hkv, q, h, &hl)) continue;
              for (int64_t e = 0; e < D; ++e) {
                int64_t from = kvslot_at(L, o, l + 1, c) + (((sp * ps + s) * Hkv + h) * D + e) * 2;
                int64_t to = kvslot_at(L, q, l, c) + (((dp * ps + s) * h_tp + hl) * D + e) * 2;
                copy2(src, dst, from, to);
              }
            }
      }
    }
  }
  return 0;
}

/* KV TP -> EP: every EP element of every live token is read from the lowest
 * TP rank holding its head (R-4) and written to the new owner's EP page.
 * Layers descending. */
uint32_t orc_kv_tp2ep(const uint8_t *src, uint8_t *dst, const int64_t *d, int64_t R, int64_t maxp,
                      const int32_t *lens, const int32_t *owner,
                      const int32_t *ep_pt, const int32_t *tp_pt, int order) {
  uint32_t flags = orc_kv_validate(d, 1, R, maxp, lens, owner, ep_pt, tp_pt);
  if (flags) return flags;
  int64_t L[OL_COUNT];
  orc_layout(d, L);
  int64_t P = d[OD_P], N = d[OD_N], Hkv = d[OD_HKV], D = d[OD_HD], ps = d[OD_PS];
  int64_t h_tp = L[OL_H_TP];
  for (int64_t t = 0; t < N; ++t) {
    int64_t l = (order < 0) ? N - 1 - t : t;
#pragma omp parallel for num_threads(g_threads) schedule(dynamic, 1) if (g_threads > 1)
    for (int64_t k = 0; k < R; ++k) {
      int64_t o = owner[k];
      for (int64_t tok = 0; tok < lens[k]; ++tok) {
        int64_t p = tok / ps, s = tok % ps;
        int64_t sp = tp_pt[k * maxp + p], dp = ep_pt[k * maxp + p];
        for (int64_t c = 0; c < 2; ++c)
          for (int64_t h = 0; h < Hkv; ++h) {
            int64_t q = 0, hl = 0;
            while (!holds_head(P, Hkv, q, h, &hl)) ++q;   /* lowest replica */
            for (int64_t e = 0; e < D; ++e) {
              int64_t from = kvslot_at(L, q, l, c) + (((sp * ps + s) * h_tp + hl) * D + e) * 2;
              int64_t to = kvslot_at(L, o, l + 1, c) + (((dp * ps + s) * Hkv + h) * D + e) * 2;
              copy2(src, dst, from, to);
            }
          }
      }
    }
  }
  return 0;
}

/* Byte offsets of one KV element in the EP and TP views (sampled checks):
 * request data (token tok of a request whose EP page is ep_page and TP page is
 * tp_page), half c, head h, dim e; TP offset for rank q (must hold h). */
void orc_kv_elem(const int64_t *d, int64_t owner, int64_t q, int64_t ep_page, int64_t tp_page,
                 int64_t tok_in_page, int64_t c, int64_t h, int64_t e,
                 int64_t ep_slot, int64_t tp_slot, int64_t *ep_off, int64_t *tp_off) {
  int64_t L[OL_COUNT];
  orc_layout(d, L);
  int64_t P = d[OD_P], Hkv = d[OD_HKV], D = d[OD_HD], ps = d[OD_PS];
  int64_t hl = -1;
  if (!holds_head(P, Hkv, q, h, &hl)) { *ep_off = -1; *tp_off = -1; return; }
  *ep_off = kvslot_at(L, owner, ep_slot, c) + (((ep_page * ps + tok_in_page) * Hkv + h) * D + e) * 2;
  *tp_off = kvslot_at(L, q, tp_slot, c) + (((tp_page * ps + tok_in_page) * L[OL_H_TP] + hl) * D + e) * 2;
}

/* ------------------------------------------------------------------------ */
/* Attention weights (memory-saving variant of §3.1)                          */
/* ------------------------------------------------------------------------ */

static int64_t attn_at(const int64_t *L, int64_t r, int64_t s) {
  return r * L[OL_REGION_STRIDE] + L[OL_ATTNSLOTS_OFF] + s * L[OL_ATTN_STRIDE];
}

/* R-16: the full-layout head held at local head slot b of TP rank q. */
static int64_t full_head_of(int64_t P, int64_t Hq, int64_t Hkv, int64_t q, int64_t b) {
  int64_t hq = Hq / P, h_tp = (Hkv >= P) ? Hkv / P : 1;
  if (b < hq) return q * hq + b;                                  /* query head */
  int64_t kv = (b - hq) % h_tp, which = (b - hq) / h_tp;         /* 0 = K, 1 = V */
  int64_t h = (Hkv >= P) ? q * h_tp + kv : q * Hkv / P;
  return Hq + which * Hkv + h;
}

/* EP -> TP: every rank keeps its own shard of its own full copy (no rank's
 * data crosses to another).  Layers ascending: EP slot l+1 -> TP slot l. */
void orc_attn_ep2tp(const uint8_t *src, uint8_t *dst, const int64_t *d, int order) {
  int64_t L[OL_COUNT];
  orc_layout(d, L);
  int64_t P = d[OD_P], H = d[OD_H], N = d[OD_N], Hkv = d[OD_HKV], D = d[OD_HD], Hq = d[OD_HQ];
  int64_t hq = Hq / P, h_tp = L[OL_H_TP];
  for (int64_t t = 0; t < N; ++t) {
    int64_t l = (order >= 0) ? t : N - 1 - t;
    for (int64_t q = 0; q < P; ++q) {
      for (int64_t b = 0; b < hq + 2 * h_tp; ++b) {
        int64_t hh = full_head_of(P, Hq, Hkv, q, b);
        for (int64_t i = 0; i < D * H; ++i)
          copy2(src, dst, attn_at(L, q, l + 1) + (hh * D * H + i) * 2, attn_at(L, q, l) + (b * D * H + i) * 2);
      }
      for (int64_t row = 0; row < H; ++row)
        for (int64_t c = 0; c < hq * D; ++c)
          copy2(src, dst, attn_at(L, q, l + 1) + L[OL_ATTN_WO_OFF] + (row * Hq * D + q * hq * D + c) * 2,
                attn_at(L, q, l) + L[OL_ATTN_WO_OFF] + (row * hq * D + c) * 2);
    }
  }
}

/* TP -> EP (all-gather): every rank's full copy is rebuilt from the shards:
 * query head hh from rank hh / (Hq/P); key or value head h from the lowest
 * rank holding it (R-4); Wo column j from rank j / ((Hq/P) * Dh).  Layers
 * descending: TP slot l -> EP slot l+1. */
void orc_attn_tp2ep(const uint8_t *src, uint8_t *dst, const int64_t *d, int order) {
  int64_t L[OL_COUNT];
  orc_layout(d, L);
  int64_t P = d[OD_P], H = d[OD_H], N = d[OD_N], Hkv = d[OD_HKV], D = d[OD_HD], Hq = d[OD_HQ];
  int64_t hq = Hq / P, h_tp = L[OL_H_TP];
  for (int64_t t = 0; t < N; ++t) {
    int64_t l = (order < 0) ? N - 1 - t : t;
    for (int64_t r = 0; r < P; ++r) {
      for (int64_t hh = 0; hh < Hq + 2 * Hkv; ++hh) {
        int64_t q, b;
        if (hh < Hq) {
          q = hh / hq;
          b = hh % hq;
        } else {
          int64_t which = (hh - Hq) / Hkv, h = (hh - Hq) % Hkv, hl = 0;
          q = 0;
          while (!holds_head(P, Hkv, q, h, &hl)) ++q;
          b = hq + which * h_tp + hl;
        }
        for (int64_t i = 0; i < D * H; ++i)
          copy2(src, dst, attn_at(L, q, l) + (b * D * H + i) * 2, attn_at(L, r, l + 1) + (hh * D * H + i) * 2);
      }
      for (int64_t row = 0; row < H; ++row)
        for (int64_t j = 0; j < Hq * D; ++j) {
          int64_t q = j / (hq * D), c = j % (hq * D);
          copy2(src, dst, attn_at(L, q, l) + L[OL_ATTN_WO_OFF] + (row * hq * D + c) * 2,
                attn_at(L, r, l + 1) + L[OL_ATTN_WO_OFF] + (row * Hq * D + j) * 2);
        }
    }
  }
}

/* ------------------------------------------------------------------------ */
/* Requests                                                                  */
/* ------------------------------------------------------------------------ */

/* §3.2 EP->TP: the ordered in-flight list every rank builds from the metadata
 * all-gather = rank 0's requests, then rank 1's, ...; inside a rank, its own
 * order (ascending request index, R-6).  tp_pos[k] = position of request k. */
void orc_request_order(int64_t P, int64_t R, const int32_t *owner, int32_t *tp_pos) {
  int64_t pos = 0;
  for (int64_t r = 0; r < P; ++r)
    for (int64_t k = 0; k < R; ++k)
      if (owner[k] == r) tp_pos[k] = (int32_t)pos++;
}

typedef struct { int64_t len, key, k; } orc_item;
static int by_len_desc_key_asc(const void *a, const void *b) {
  const orc_item *x = a, *y = b;
  if (x->len != y->len) return x->len > y->len ? -1 : 1;
  if (x->key != y->key) return x->key < y->key ? -1 : 1;
  return 0;
}

/* §3.2 TP->EP placement: sort the global list by length, longest first (ties:
 * list position), then give each request to the rank with the smallest load
 * so far (ties: lowest rank); load = tokens (R-5).  local_pos = rank of the
 * request among its owner's requests by list position (R-6).  key == NULL
 * means list position = request index.  Returns the max load. */
int64_t orc_place(int64_t P, int64_t R, const int32_t *lens, const int32_t *key,
                  int32_t *owner, int32_t *local_pos) {
  orc_item *it = malloc(sizeof(orc_item) * (size_t)(R > 0 ? R : 1));
  int64_t *load = calloc((size_t)P, sizeof(int64_t));
  for (int64_t k = 0; k < R; ++k) {
    it[k].len = lens[k];
    it[k].key = key ? key[k] : k;
    it[k].k = k;
  }
  qsort(it, (size_t)R, sizeof(orc_item), by_len_desc_key_asc);
  for (int64_t n = 0; n < R; ++n) {
    int64_t best = 0;
    for (int64_t q = 1; q < P; ++q)
      if (load[q] < load[best]) best = q;
    owner[it[n].k] = (int32_t)best;
    load[best] += it[n].len;
  }
  for (int64_t k = 0; k < R; ++k) {
    int64_t kk = key ? key[k] : k, cnt = 0;
    for (int64_t m = 0; m < R; ++m) {
      int64_t km = key ? key[m] : m;
      if (owner[m] == owner[k] && km < kk) ++cnt;
    }
    local_pos[k] = (int32_t)cnt;
  }
  int64_t mx = 0;
  for (int64_t q = 0; q < P; ++q)
    if (load[q] > mx) mx = load[q];
  free(load);
  free(it);
  return mx;
}

/* R-7: page hand-out.  Pool g (= region[k], or pool 0 when region == NULL)
 * gives its free pages free_pages[g*free_stride + 0 ..] to its requests in
 * ascending key order (key == NULL: request index), each request taking
 * ceil(len/ps) consecutive entries.  Rows are filled with -1 past the
 * request's pages.  On shortage nothing is written and ORC_F_CAPACITY is
 * returned; a bad length or region gives ORC_F_BAD_REQUEST. */
uint32_t orc_assign_pages(int64_t npools, int64_t R, int64_t ps, int64_t maxp,
                          const int32_t *lens, const int32_t *region, const int32_t *key,
                          const int32_t *free_pages, int64_t free_stride, int64_t free_count,
                          int32_t *pt) {
  for (int64_t k = 0; k < R; ++k) {
    int64_t g = region ? region[k] : 0;
    if (lens[k] < 0 || (int64_t)lens[k] > maxp * ps || g < 0 || g >= npools) return ORC_F_BAD_REQUEST;
  }
  int64_t *start = malloc(sizeof(int64_t) * (size_t)(R > 0 ? R : 1));
  for (int64_t k = 0; k < R; ++k) {
    int64_t g = region ? region[k] : 0, kk = key ? key[k] : k, s = 0;
    for (int64_t m = 0; m < R; ++m) {
      int64_t gm = region ? region[m] : 0, km = key ? key[m] : m;
      if (gm == g && km < kk) s += npages_of(lens[m], ps);
    }
    start[k] = s;
    if (s + npages_of(lens[k], ps) > free_count) { free(start); return ORC_F_CAPACITY; }
  }
  for (int64_t k = 0; k < R; ++k) {
    int64_t g = region ? region[k] : 0, np = npages_of(lens[k], ps);
    for (int64_t p = 0; p < maxp; ++p)
      pt[k * maxp + p] = (p < np) ? free_pages[g * free_stride + start[k] + p] : -1;
  }
  free(start);
  return 0;
}

/* §4.3: page-indexed work descriptors, one per (request, logical page), grouped
 * by the rank whose bytes they move (EP->TP: the EP owner the page is read
 * from; TP->EP: the EP owner it is written to), then by request, then page.
 * Each record is 8 int32: request, page, src rank (-1 = per head), dst rank
 * (-1 = every holder), src page, dst page, tokens, 0.  Returns the count. */
int64_t orc_kv_descriptors(const int64_t *d, int dir, int64_t R, int64_t maxp,
                           const int32_t *lens, const int32_t *owner,
                           const int32_t *ep_pt, const int32_t *tp_pt, int32_t *out) {
  int64_t P = d[OD_P], ps = d[OD_PS], n = 0;
  for (int64_t r = 0; r < P; ++r)
    for (int64_t k = 0; k < R; ++k) {
      if (owner[k] != r) continue;
      int64_t np = npages_of(lens[k], ps);
      for (int64_t p = 0; p < np; ++p) {
        int32_t *o = out + 8 * n;
        o[0] = (int32_t)k;
        o[1] = (int32_t)p;
        o[2] = dir == 0 ? (int32_t)r : -1;
        o[3] = dir == 0 ? -1 : (int32_t)r;
        o[4] = dir == 0 ? ep_pt[k * maxp + p] : tp_pt[k * maxp + p];
        o[5] = dir == 0 ? tp_pt[k * maxp + p] : ep_pt[k * maxp + p];
        o[6] = (int32_t)(lens[k] - p * ps < ps ? lens[k] - p * ps : ps);
        o[7] = 0;
        ++n;
      }
    }
  return n;
}
