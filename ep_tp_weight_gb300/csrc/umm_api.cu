// C ABI of libumm: handle, layout of the unified buffer, argument checks,
// modes, status and per-kernel timing.  Kernels live in umm_weights.cu
// (expert weights), umm_kv_prep.cu and umm_kv.cu (KV descriptor pass and
// copies), umm_kv_staged.cu (staged KV path), umm_attn.cu (attention weights)
// and umm_requests.cu (request order, placement, page hand-out).
//
// Layout (unified memory manager of "Moebius: Serving Mixture-of-Expert Models
// with Seamless Runtime Parallelism Switch" (paper review), §4.2, Fig. 7): one
// region per rank = N+1 weight slots, N+1 KV slots, then N+1 attention slots;
// TP layer l in slot l, EP layer l in slot l+1; a workspace after the P
// regions.
#include <algorithm>
#include <cstdio>
#include <cstring>
#include <new>
#include <vector>

#include "umm_internal.cuh"

namespace {

constexpr uint64_t kStatusBytes = 256;

uint64_t align_up(uint64_t x, uint64_t a) { return (x + a - 1) / a * a; }

struct Prof {
  int kind;
  int units;   // layer copies (copy kinds) or calls (metadata kinds) timed
  cudaEvent_t a, b;
};

struct KvCall {
  unsigned int id;
  int32_t mode_before;
};

}  // namespace

struct umm {
  umm_dims dims;
  umm_layout_t L;
  uk::Geo geo;
  uk::Ws ws;
  int device = 0;
  int sms = 1;
  int32_t weight_mode = UMM_MODE_EP, kv_mode = UMM_MODE_EP, attn_mode = UMM_MODE_EP;
  unsigned int next_call = 0;
  std::vector<KvCall> kv_log;
  bool prof = false;
  std::vector<cudaEvent_t> ev_pool;
  std::vector<Prof> pending;
  int64_t launches = 0;   // kernels enqueued by this handle
  int64_t prof_n[UMM_K_COUNT] = {};
  double prof_ms[UMM_K_COUNT] = {};
  // opt-in (umm_set_switch_overlap): the weight reshards of a one-call switch
  // run on a side stream, beside the request bookkeeping and the KV reshard
  bool overlap = false;
  cudaStream_t side = nullptr;
  cudaEvent_t ev_fork = nullptr, ev_join = nullptr;
  // umm_test_stall_tma_wait (checked build): the KV EP->TP layer whose TMA
  // copy makes one wait that runs out after test_stall_polls polls
  int32_t test_stall_layer = -1;
  uint32_t test_stall_polls = 0;
};

namespace {

int check_dims(const umm_dims* d) {
  if (!d) return UMM_ERR_INVALID_ARG;
  if (d->P < 1 || d->P > uk::kMaxGroups || d->num_layers < 1 || d->num_layers > 4096) return UMM_ERR_INVALID_ARG;
  if (d->E < 0 || d->E % d->P) return UMM_ERR_INVALID_ARG;
  if (d->E > 0) {
    if (d->H < 1 || d->I < 1 || d->I % d->P) return UMM_ERR_INVALID_ARG;
    const uint64_t el = (uint64_t)(d->E / d->P);
    // per-region element count must stay addressable by 32-bit vector indices
    if (el * 3ull * (uint64_t)d->I * (uint64_t)d->H >= (1ull << 31) - (1ull << 16)) return UMM_ERR_INVALID_ARG;
  }
  if (d->num_kv_heads < 0) return UMM_ERR_INVALID_ARG;
  if (d->num_kv_heads > 0) {
    const int hkv = d->num_kv_heads, P = d->P;
    if (hkv % P != 0 && P % hkv != 0) return UMM_ERR_INVALID_ARG;
    if (d->head_dim < 1 || d->page_size < 1 || d->kv_pages_tp < 1) return UMM_ERR_INVALID_ARG;
    const int64_t h_tp = hkv >= P ? hkv / P : 1;
    if (d->kv_pages_tp % (hkv / h_tp)) return UMM_ERR_INVALID_ARG;
    if (d->kv_pages_tp >= (1ll << 31)) return UMM_ERR_INVALID_ARG;
    if ((uint64_t)d->page_size * hkv * d->head_dim * 2 >= (1ull << 30)) return UMM_ERR_INVALID_ARG;
  }
  if (d->max_requests < 0 || d->max_requests > (1 << 26)) return UMM_ERR_INVALID_ARG;
  if (d->max_pages < 0 || d->max_pages >= (1ll << 31)) return UMM_ERR_INVALID_ARG;
  if (d->w13_split != 0 && d->w13_split != 1) return UMM_ERR_INVALID_ARG;
  if ((d->weight_mode != UMM_MODE_EP && d->weight_mode != UMM_MODE_TP) ||
      (d->kv_mode != UMM_MODE_EP && d->kv_mode != UMM_MODE_TP) ||
      (d->attn_mode != UMM_MODE_EP && d->attn_mode != UMM_MODE_TP))
    return UMM_ERR_INVALID_ARG;
  if (d->attn_q_heads < 0) return UMM_ERR_INVALID_ARG;
  if (d->attn_q_heads > 0) {
    if (d->num_kv_heads < 1 || d->head_dim < 1 || d->H < 1 || d->attn_q_heads % d->P) return UMM_ERR_INVALID_ARG;
    const uint64_t hq = (uint64_t)(d->attn_q_heads / d->P);
    const uint64_t h_tp = (uint64_t)(d->num_kv_heads >= d->P ? d->num_kv_heads / d->P : 1);
    // per-rank shard element count must stay addressable by 32-bit vector indices
    if ((hq + 2 * h_tp) * d->head_dim * (uint64_t)d->H + (uint64_t)d->H * hq * d->head_dim >= (1ull << 31) - (1ull << 16))
      return UMM_ERR_INVALID_ARG;
  }
  return UMM_OK;
}

// Layout: region = [weight slot 0..N][KV slot 0..N][attention slot 0..N]; W2 at 256 B inside a
// weight slot, V at 256 B after K inside a KV slot, slot strides rounded to
// 4 KiB, region stride to 2 MiB; workspace after the last region.
void compute_layout(const umm_dims* d, umm_layout_t* L, uk::Ws* ws) {
  std::memset(L, 0, sizeof(*L));
  const uint64_t P = d->P, N = d->num_layers;
  const uint64_t El = d->E > 0 ? (uint64_t)(d->E / d->P) : 0;
  const uint64_t w13 = El * 2ull * d->I * d->H * 2ull;
  const uint64_t w2 = El * (uint64_t)d->H * d->I * 2ull;
  L->w13_off = 0;
  L->w2_off = align_up(w13, 256);
  L->wslot_stride = d->E > 0 ? align_up(L->w2_off + w2, 4096) : 0;
  const int64_t hkv = d->num_kv_heads;
  L->h_tp = hkv > 0 ? (hkv >= d->P ? hkv / d->P : 1) : 0;
  L->pages_tp = hkv > 0 ? d->kv_pages_tp : 0;
  L->pages_ep = hkv > 0 ? d->kv_pages_tp * L->h_tp / hkv : 0;
  const uint64_t half = hkv > 0 ? (uint64_t)L->pages_tp * d->page_size * L->h_tp * d->head_dim * 2ull : 0;
  L->kv_v_off = align_up(half, 256);
  L->kvslot_stride = hkv > 0 ? align_up(L->kv_v_off + half, 4096) : 0;
  L->kvslots_off = (N + 1) * L->wslot_stride;
  // attention slots (memory-saving variant), sized for the full EP copy
  const uint64_t hq = (uint64_t)d->attn_q_heads;
  const uint64_t qkv = hq > 0 ? (hq + 2ull * (uint64_t)hkv) * d->head_dim * (uint64_t)d->H * 2ull : 0;
  L->attn_wo_off = align_up(qkv, 256);
  L->attnslot_stride = hq > 0 ? align_up(L->attn_wo_off + (uint64_t)d->H * hq * d->head_dim * 2ull, 4096) : 0;
  L->attnslots_off = (N + 1) * (L->wslot_stride + L->kvslot_stride);
  L->region_stride = align_up((N + 1) * (L->wslot_stride + L->kvslot_stride + L->attnslot_stride), 2ull << 20);
  L->ws_off = P * L->region_stride;

  const int64_t desc_cap = d->max_pages > 0 ? d->max_pages : L->pages_tp;
  const int64_t nreq = d->max_requests > 0 ? d->max_requests : 1;
  int64_t keys_cap = 1;
  while (keys_cap < nreq) keys_cap <<= 1;
  const int64_t bits = std::max<int64_t>(L->pages_tp, (int64_t)P * L->pages_ep);
  const int64_t words = (bits + 31) / 32 + 1;
  uint64_t o = L->ws_off;
  ws->status = o;
  o += kStatusBytes;
  ws->desc = o;
  ws->desc_cap = desc_cap;
  o = align_up(o + (uint64_t)desc_cap * sizeof(umm_kv_desc), 256);
  ws->req_off = o;
  o = align_up(o + (uint64_t)nreq * 8, 256);
  ws->req_inv = o;
  o = align_up(o + (uint64_t)nreq * 4, 256);
  ws->keys = o;
  ws->keys_cap = keys_cap;
  o = align_up(o + (uint64_t)keys_cap * 8, 256);
  ws->choice = o;
  o = align_up(o + (uint64_t)nreq + 4, 256);
  ws->bitmap = o;
  ws->bitmap_words = words;
  o = align_up(o + (uint64_t)words * 4, 256);
  ws->tp_bitmap = o;
  o = align_up(o + (uint64_t)((L->pages_tp + 31) / 32 + 1) * 4, 256);
  ws->sched = o;
  o = align_up(o + (uint64_t)L->pages_tp * 8, 256);
  ws->order_tok = o;
  o = align_up(o + (uint64_t)nreq * 8, 256);
  ws->rank_info = o;
  o = align_up(o + (uint64_t)3 * uk::kMaxGroups * 8, 4096);
  ws->max_requests = (int32_t)nreq;
  L->ws_bytes = o - L->ws_off;
  L->total_bytes = o;
  L->status_off = ws->status;
  L->desc_off = ws->desc;
  L->desc_capacity = desc_cap;
}

// What the kernels need to address a buffer at `base` laid out as L.
uk::Geo make_geo(const umm_dims* dims, const umm_layout_t& L, const uk::Ws& ws, uint8_t* base) {
  uk::Geo g;
  g.base = base;
  g.region_stride = L.region_stride;
  g.wslot_stride = L.wslot_stride;
  g.w13_off = L.w13_off;
  g.w2_off = L.w2_off;
  g.kvslot_stride = L.kvslot_stride;
  g.kv_v_off = L.kv_v_off;
  g.kvslots_off = L.kvslots_off;
  g.P = dims->P;
  g.E = dims->E;
  g.H = dims->H;
  g.I = dims->I;
  g.N = dims->num_layers;
  g.Hkv = dims->num_kv_heads;
  g.D = dims->head_dim;
  g.ps = dims->page_size;
  g.w13_split = dims->w13_split;
  g.Hq = dims->attn_q_heads;
  g.attnslot_stride = L.attnslot_stride;
  g.attn_wo_off = L.attn_wo_off;
  g.attnslots_off = L.attnslots_off;
  g.flags = base ? reinterpret_cast<unsigned int*>(base + ws.status) : nullptr;
  g.pages_ep = L.pages_ep;
  g.pages_tp = L.pages_tp;
  g.h_tp = L.h_tp;
  return g;
}

cudaStream_t as_stream(void* s) { return reinterpret_cast<cudaStream_t>(s); }

unsigned int new_call(umm* u) {
  if (++u->next_call == 0) u->next_call = 1;
  return u->next_call;
}

// ---- per-kernel event timing ----
// One event pair per scope.  The layer copies of one call sit in one scope
// (units = their number), so the events never break their launch chain.
struct ProfScope {
  umm* u;
  int kind;
  cudaStream_t s;
  int units = 1;
  cudaEvent_t a = nullptr, b = nullptr;
  ProfScope(umm* uu, int k, cudaStream_t ss) : u(uu), kind(k), s(ss) {
    if (!u->prof || u->ev_pool.size() < 2) return;
    b = u->ev_pool.back();
    u->ev_pool.pop_back();
    a = u->ev_pool.back();
    u->ev_pool.pop_back();
    cudaEventRecord(a, s);
  }
  ~ProfScope() {
    if (!a) return;
    cudaEventRecord(b, s);
    u->pending.push_back(Prof{kind, units, a, b});
  }
};

int cuda_rc(cudaError_t e) { return e == cudaSuccess ? UMM_OK : UMM_ERR_CUDA; }

// Layer t of a call's copies runs as a programmatic dependent of layer t-1
// (launch_chain); per-kernel timing brackets the whole chain (ProfScope).
bool chained(int t) { return t > 0; }

int check_kv_args(const umm* u, int32_t R, int32_t maxp, const void* a, const void* b, const void* c,
                  const void* d) {
  if (!u || u->dims.num_kv_heads == 0) return UMM_ERR_INVALID_ARG;
  if (R < 0 || R > u->ws.max_requests || maxp < 1) return UMM_ERR_INVALID_ARG;
  if ((int64_t)maxp * u->dims.page_size > 0x7fffffffll) return UMM_ERR_INVALID_ARG;
  if (R > 0 && (!a || !b || !c || !d)) return UMM_ERR_INVALID_ARG;
  return UMM_OK;
}

// tma: the EP->TP copy may run through TMA (kv_copy_ep2tp_tma).  A one-call
// switch that runs the weight copies beside the KV (side stream) passes
// false: beside them the LSU copy measured faster on GB300 (16 requests:
// 6.15 vs 6.32 ms per round trip; 2048 requests: equal), while alone TMA is
// faster.
int reshard_kv(umm* u, int dir, int32_t R, int32_t maxp, const int32_t* lens, const int32_t* owner,
               const int32_t* ep_pt, const int32_t* tp_pt, void* stream, bool tma = true) {
  int rc = check_kv_args(u, R, maxp, lens, owner, ep_pt, tp_pt);
  if (rc) return rc;
  const int32_t from = dir == 0 ? UMM_MODE_EP : UMM_MODE_TP;
  if (u->kv_mode != from) return UMM_ERR_MODE;
  cudaStream_t s = as_stream(stream);
  const unsigned int call = new_call(u);
  // live pages <= min(descriptor capacity, R * pages per request).  When they
  // may fill half the TP pool or more, the copies walk the pool in TP-page
  // order (measured on GB300: +1.7% EP->TP, +2.3% TP->EP over list order).
  const int64_t max_desc = std::min<int64_t>(u->ws.desc_cap, (int64_t)R * maxp);
  const int use_sched = max_desc > 0 && 2 * max_desc >= u->L.pages_tp;
  {
    ProfScope ps(u, UMM_K_KV_PREP, s);
    rc = cuda_rc(uk::launch_kv_prep(u->geo, u->ws, dir, R, maxp, lens, owner, ep_pt, tp_pt, call, use_sched, s,
                                    u->sms));
  }
  if (rc) return rc;
  u->launches += R > 0 ? 2 : 1;
  const int N = u->dims.num_layers;
  {
    ProfScope ps(u, dir == 0 ? UMM_K_KV_EP2TP : UMM_K_KV_TP2EP, s);
    ps.units = max_desc > 0 ? N : 0;
    for (int t = 0; t < N; ++t) {
      const int layer = dir == 0 ? t : N - 1 - t;   // EP->TP ascending, TP->EP descending
      const uint32_t stall = dir == 0 && layer == u->test_stall_layer ? u->test_stall_polls : 0u;
      rc = cuda_rc(
          uk::launch_kv_copy(u->geo, u->ws, dir, layer, max_desc, use_sched, call, s, chained(t), tma, stall));
      if (rc) return rc;
      if (max_desc > 0) ++u->launches;
    }
  }
  u->kv_log.push_back(KvCall{call, u->kv_mode});
  if (u->kv_log.size() > 4096) u->kv_log.erase(u->kv_log.begin());
  u->kv_mode = dir == 0 ? UMM_MODE_TP : UMM_MODE_EP;
  return UMM_OK;
}

int reshard_weights(umm* u, int ep2tp, void* stream) {
  if (!u || u->dims.E == 0) return UMM_ERR_INVALID_ARG;
  if (u->weight_mode != (ep2tp ? UMM_MODE_EP : UMM_MODE_TP)) return UMM_ERR_MODE;
  cudaStream_t s = as_stream(stream);
  const int N = u->dims.num_layers;
  ProfScope ps(u, ep2tp ? UMM_K_WEIGHTS_EP2TP : UMM_K_WEIGHTS_TP2EP, s);
  ps.units = N;
  for (int t = 0; t < N; ++t) {
    const int layer = ep2tp ? t : N - 1 - t;
    int rc = cuda_rc(uk::launch_weights(u->geo, ep2tp, layer, s, chained(t)));
    if (rc) return rc;
    ++u->launches;
  }
  u->weight_mode = ep2tp ? UMM_MODE_TP : UMM_MODE_EP;
  return UMM_OK;
}

int reshard_kv_staged(umm* u, int dir, void* d_stage, uint64_t stage_bytes, int32_t R, int32_t maxp,
                      const int32_t* lens, const int32_t* owner, const int32_t* ep_pt, const int32_t* tp_pt,
                      void* stream) {
  int rc = check_kv_args(u, R, maxp, lens, owner, ep_pt, tp_pt);
  if (rc) return rc;
  if (!d_stage) return UMM_ERR_INVALID_ARG;
  if (reinterpret_cast<uintptr_t>(d_stage) % 256) return UMM_ERR_ALIGN;
  if (stage_bytes < uk::kv_stage_bytes(u->geo)) return UMM_ERR_CAPACITY;
  if (u->kv_mode != (dir == 0 ? UMM_MODE_EP : UMM_MODE_TP)) return UMM_ERR_MODE;
  cudaStream_t s = as_stream(stream);
  const unsigned int call = new_call(u);
  {
    ProfScope ps(u, UMM_K_KV_PREP, s);
    rc = cuda_rc(uk::launch_kv_prep(u->geo, u->ws, dir, R, maxp, lens, owner, ep_pt, tp_pt, call, 0, s, u->sms));
  }
  if (rc) return rc;
  u->launches += R > 0 ? 2 : 1;
  {
    ProfScope ps(u, dir == 0 ? UMM_K_KV_EP2TP : UMM_K_KV_TP2EP, s);
    ps.units = u->dims.num_layers;
    int n = 0;
    rc = cuda_rc(uk::launch_kv_staged(u->geo, u->ws, dir, R, lens, owner, static_cast<uint8_t*>(d_stage),
                                      reinterpret_cast<int64_t*>(u->geo.base + u->ws.order_tok),
                                      reinterpret_cast<int64_t*>(u->geo.base + u->ws.rank_info), call, s, u->sms,
                                      &n));
    u->launches += n;
  }
  if (rc) return rc;
  u->kv_log.push_back(KvCall{call, u->kv_mode});
  if (u->kv_log.size() > 4096) u->kv_log.erase(u->kv_log.begin());
  u->kv_mode = dir == 0 ? UMM_MODE_TP : UMM_MODE_EP;
  return UMM_OK;
}

int reshard_weights_staged(umm* u, int ep2tp, void* d_stage, uint64_t stage_bytes, void* stream) {
  if (!u || u->dims.E == 0 || !d_stage) return UMM_ERR_INVALID_ARG;
  if (reinterpret_cast<uintptr_t>(d_stage) % 256) return UMM_ERR_ALIGN;
  if (stage_bytes < uk::weights_stage_bytes(u->geo)) return UMM_ERR_CAPACITY;
  if (u->weight_mode != (ep2tp ? UMM_MODE_EP : UMM_MODE_TP)) return UMM_ERR_MODE;
  cudaStream_t s = as_stream(stream);
  const int N = u->dims.num_layers;
  for (int t = 0; t < N; ++t) {
    const int layer = ep2tp ? t : N - 1 - t;
    ProfScope ps(u, ep2tp ? UMM_K_WEIGHTS_EP2TP : UMM_K_WEIGHTS_TP2EP, s);
    int n = 0;
    int rc = cuda_rc(uk::launch_weights_staged(u->geo, ep2tp, layer, static_cast<uint8_t*>(d_stage), s, &n));
    if (rc) return rc;
    u->launches += n;
  }
  u->weight_mode = ep2tp ? UMM_MODE_TP : UMM_MODE_EP;
  return UMM_OK;
}

}  // namespace

extern "C" {

int umm_required_bytes(const umm_dims* dims, uint64_t* bytes_out) {
  int rc = check_dims(dims);
  if (rc) return rc;
  if (!bytes_out) return UMM_ERR_INVALID_ARG;
  umm_layout_t L;
  uk::Ws ws;
  compute_layout(dims, &L, &ws);
  *bytes_out = L.total_bytes;
  return UMM_OK;
}

int umm_layout_for_dims(const umm_dims* dims, umm_layout_t* out) {
  int rc = check_dims(dims);
  if (rc) return rc;
  if (!out) return UMM_ERR_INVALID_ARG;
  uk::Ws ws;
  compute_layout(dims, out, &ws);
  return UMM_OK;
}

int umm_kv_copy_kernel(const umm_dims* dims, int32_t dir, int32_t* kernel, int32_t* vector_bytes) {
  int rc = check_dims(dims);
  if (rc) return rc;
  if (dims->num_kv_heads == 0 || (dir != 0 && dir != 1) || !kernel) return UMM_ERR_INVALID_ARG;
  umm_layout_t L;
  uk::Ws ws;
  compute_layout(dims, &L, &ws);
  const uk::Geo g = make_geo(dims, L, ws, nullptr);
  const bool tma = dir == 0 && uk::ep2tp_tma_shape(g);
  *kernel = tma ? UMM_KV_COPY_TMA : UMM_KV_COPY_LSU;
  if (vector_bytes) *vector_bytes = tma ? 0 : uk::kv_vector_bytes(g);
  return UMM_OK;
}

int umm_create(const umm_dims* dims, void* d_base, uint64_t bytes, umm_t** out) {
  int rc = check_dims(dims);
  if (rc) return rc;
  if (!out || !d_base) return UMM_ERR_INVALID_ARG;
  if (reinterpret_cast<uintptr_t>(d_base) % 256) return UMM_ERR_ALIGN;
  umm* u = new (std::nothrow) umm();
  if (!u) return UMM_ERR_INVALID_ARG;
  u->dims = *dims;
  if (u->dims.max_pages == 0) u->dims.max_pages = dims->num_kv_heads > 0 ? dims->kv_pages_tp : 0;
  compute_layout(&u->dims, &u->L, &u->ws);
  if (bytes < u->L.total_bytes) {
    delete u;
    return UMM_ERR_CAPACITY;
  }
  cudaPointerAttributes attr;
  if (cudaPointerGetAttributes(&attr, d_base) != cudaSuccess || attr.type != cudaMemoryTypeDevice) {
    cudaGetLastError();
    delete u;
    return UMM_ERR_INVALID_ARG;
  }
  u->device = attr.device;
  int dev_now = 0;
  cudaGetDevice(&dev_now);
  if (dev_now != u->device) {
    delete u;
    return UMM_ERR_INVALID_ARG;
  }
  cudaDeviceGetAttribute(&u->sms, cudaDevAttrMultiProcessorCount, u->device);
  if (u->sms < 1) u->sms = 1;
  u->geo = make_geo(dims, u->L, u->ws, static_cast<uint8_t*>(d_base));
  uk::Geo& g = u->geo;
  u->weight_mode = dims->weight_mode;
  u->kv_mode = dims->kv_mode;
  u->attn_mode = dims->attn_mode;
  // status block and TP-page schedule start at zero (call id 0 is never used)
  if (cudaMemset(g.base + u->ws.status, 0, kStatusBytes) != cudaSuccess ||
      (u->L.pages_tp > 0 && cudaMemset(g.base + u->ws.sched, 0, (size_t)u->L.pages_tp * 8) != cudaSuccess) ||
      cudaDeviceSynchronize() != cudaSuccess) {
    delete u;
    return UMM_ERR_CUDA;
  }
  *out = u;
  return UMM_OK;
}

int umm_destroy(umm_t* u) {
  if (!u) return UMM_ERR_INVALID_ARG;
  if (u->side) cudaStreamDestroy(u->side);   // resources go once its work is done
  if (u->ev_fork) cudaEventDestroy(u->ev_fork);
  if (u->ev_join) cudaEventDestroy(u->ev_join);
  for (auto& p : u->pending) {
    cudaEventDestroy(p.a);
    cudaEventDestroy(p.b);
  }
  for (auto e : u->ev_pool) cudaEventDestroy(e);
  delete u;
  return UMM_OK;
}

int umm_layout(const umm_t* u, umm_layout_t* out) {
  if (!u || !out) return UMM_ERR_INVALID_ARG;
  *out = u->L;
  return UMM_OK;
}

int umm_get_modes(const umm_t* u, int32_t* weight_mode, int32_t* kv_mode) {
  if (!u) return UMM_ERR_INVALID_ARG;
  if (weight_mode) *weight_mode = u->weight_mode;
  if (kv_mode) *kv_mode = u->kv_mode;
  return UMM_OK;
}

int umm_set_modes(umm_t* u, int32_t weight_mode, int32_t kv_mode) {
  if (!u) return UMM_ERR_INVALID_ARG;
  if ((weight_mode != UMM_MODE_EP && weight_mode != UMM_MODE_TP) ||
      (kv_mode != UMM_MODE_EP && kv_mode != UMM_MODE_TP))
    return UMM_ERR_INVALID_ARG;
  u->weight_mode = weight_mode;
  u->kv_mode = kv_mode;
  u->kv_log.clear();
  return UMM_OK;
}

static int reshard_attn(umm_t* u, int ep2tp, void* stream) {
  if (!u || u->dims.attn_q_heads == 0) return UMM_ERR_INVALID_ARG;
  if (u->attn_mode != (ep2tp ? UMM_MODE_EP : UMM_MODE_TP)) return UMM_ERR_MODE;
  cudaStream_t s = as_stream(stream);
  const int N = u->dims.num_layers;
  ProfScope ps(u, ep2tp ? UMM_K_ATTN_EP2TP : UMM_K_ATTN_TP2EP, s);
  ps.units = N;
  for (int t = 0; t < N; ++t) {
    const int layer = ep2tp ? t : N - 1 - t;
    int rc = cuda_rc(uk::launch_attn(u->geo, ep2tp, layer, s, chained(t)));
    if (rc) return rc;
    ++u->launches;
  }
  u->attn_mode = ep2tp ? UMM_MODE_TP : UMM_MODE_EP;
  return UMM_OK;
}

int reshard_attn_ep2tp(umm_t* u, void* stream) { return reshard_attn(u, 1, stream); }
int reshard_attn_tp2ep(umm_t* u, void* stream) { return reshard_attn(u, 0, stream); }

int umm_get_attn_mode(const umm_t* u, int32_t* mode) {
  if (!u || !mode) return UMM_ERR_INVALID_ARG;
  *mode = u->attn_mode;
  return UMM_OK;
}

int umm_set_attn_mode(umm_t* u, int32_t mode) {
  if (!u || (mode != UMM_MODE_EP && mode != UMM_MODE_TP)) return UMM_ERR_INVALID_ARG;
  u->attn_mode = mode;
  return UMM_OK;
}

int reshard_weights_ep2tp(umm_t* u, void* stream) { return reshard_weights(u, 1, stream); }
int reshard_weights_tp2ep(umm_t* u, void* stream) { return reshard_weights(u, 0, stream); }

int umm_weights_stage_bytes(const umm_t* u, uint64_t* bytes_out) {
  if (!u || !bytes_out || u->dims.E == 0) return UMM_ERR_INVALID_ARG;
  *bytes_out = uk::weights_stage_bytes(u->geo);
  return UMM_OK;
}

int reshard_weights_ep2tp_staged(umm_t* u, void* d_stage, uint64_t stage_bytes, void* stream) {
  return reshard_weights_staged(u, 1, d_stage, stage_bytes, stream);
}

int reshard_weights_tp2ep_staged(umm_t* u, void* d_stage, uint64_t stage_bytes, void* stream) {
  return reshard_weights_staged(u, 0, d_stage, stage_bytes, stream);
}

int gather_requests_ep2tp(umm_t* u, int32_t R, const int32_t* d_ep_owner, int32_t* d_tp_pos, void* stream) {
  if (!u || R < 0 || R > u->ws.max_requests) return UMM_ERR_INVALID_ARG;
  if (R > 0 && (!d_ep_owner || !d_tp_pos)) return UMM_ERR_INVALID_ARG;
  if (R == 0) return UMM_OK;
  cudaStream_t s = as_stream(stream);
  const unsigned int call = new_call(u);
  ProfScope ps(u, UMM_K_ORDER, s);
  u->launches += 1;
  return cuda_rc(uk::launch_order(u->geo, u->ws, R, d_ep_owner, d_tp_pos, call, s));
}

int place_requests_tp2ep(umm_t* u, int32_t R, const int32_t* d_seq_lens, const int32_t* d_list_pos,
                         int32_t* d_owner, int32_t* d_local_pos, void* stream) {
  if (!u || R < 0 || R > u->ws.max_requests) return UMM_ERR_INVALID_ARG;
  if (R > 0 && (!d_seq_lens || !d_owner || !d_local_pos)) return UMM_ERR_INVALID_ARG;
  if (R == 0) return UMM_OK;
  cudaStream_t s = as_stream(stream);
  const unsigned int call = new_call(u);
  ProfScope ps(u, UMM_K_PLACE, s);
  u->launches += 1;
  return cuda_rc(uk::launch_place(u->geo, u->ws, R, d_seq_lens, d_list_pos, d_owner, d_local_pos, call, s));
}

int umm_assign_pages(umm_t* u, int32_t npools, int32_t R, const int32_t* d_seq_lens, const int32_t* d_pool,
                     const int32_t* d_key, const int32_t* d_free_pages, int64_t free_stride,
                     int64_t free_count, int32_t* d_page_table, int32_t max_pages_per_req, void* stream) {
  if (!u || npools < 1 || npools > uk::kMaxGroups || R < 0 || R > u->ws.max_requests) return UMM_ERR_INVALID_ARG;
  if (max_pages_per_req < 1 || free_count < 0 || (npools > 1 && free_stride < free_count))
    return UMM_ERR_INVALID_ARG;
  if ((int64_t)max_pages_per_req * (u->dims.page_size > 0 ? u->dims.page_size : 1) > 0x7fffffffll)
    return UMM_ERR_INVALID_ARG;
  if (npools > 1 && !d_pool) return UMM_ERR_INVALID_ARG;
  if (R > 0 && (!d_seq_lens || !d_free_pages || !d_page_table)) return UMM_ERR_INVALID_ARG;
  if (u->dims.page_size < 1) return UMM_ERR_INVALID_ARG;
  if (R == 0) return UMM_OK;
  cudaStream_t s = as_stream(stream);
  const unsigned int call = new_call(u);
  ProfScope ps(u, UMM_K_ASSIGN, s);
  u->launches += 2;
  return cuda_rc(uk::launch_assign(u->geo, u->ws, npools, R, d_seq_lens, d_pool, d_key, d_free_pages,
                                   free_stride, free_count, d_page_table, max_pages_per_req, call, s, u->sms));
}

int umm_kv_stage_bytes(const umm_t* u, uint64_t* bytes_out) {
  if (!u || !bytes_out || u->dims.num_kv_heads == 0) return UMM_ERR_INVALID_ARG;
  *bytes_out = uk::kv_stage_bytes(u->geo);
  return UMM_OK;
}

int reshard_kv_ep2tp_staged(umm_t* u, void* d_stage, uint64_t stage_bytes, int32_t R, int32_t max_pages_per_req,
                            const int32_t* d_seq_lens, const int32_t* d_ep_owner, const int32_t* d_ep_page_table,
                            const int32_t* d_tp_page_table, void* stream) {
  return reshard_kv_staged(u, 0, d_stage, stage_bytes, R, max_pages_per_req, d_seq_lens, d_ep_owner,
                           d_ep_page_table, d_tp_page_table, stream);
}

int reshard_kv_tp2ep_staged(umm_t* u, void* d_stage, uint64_t stage_bytes, int32_t R, int32_t max_pages_per_req,
                            const int32_t* d_seq_lens, const int32_t* d_ep_owner, const int32_t* d_ep_page_table,
                            const int32_t* d_tp_page_table, void* stream) {
  return reshard_kv_staged(u, 1, d_stage, stage_bytes, R, max_pages_per_req, d_seq_lens, d_ep_owner,
                           d_ep_page_table, d_tp_page_table, stream);
}

int reshard_kv_ep2tp(umm_t* u, int32_t R, int32_t max_pages_per_req, const int32_t* d_seq_lens,
                     const int32_t* d_ep_owner, const int32_t* d_ep_page_table,
                     const int32_t* d_tp_page_table, void* stream) {
  return reshard_kv(u, 0, R, max_pages_per_req, d_seq_lens, d_ep_owner, d_ep_page_table, d_tp_page_table,
                    stream);
}

int reshard_kv_tp2ep(umm_t* u, int32_t R, int32_t max_pages_per_req, const int32_t* d_seq_lens,
                     const int32_t* d_ep_owner, const int32_t* d_ep_page_table,
                     const int32_t* d_tp_page_table, void* stream) {
  return reshard_kv(u, 1, R, max_pages_per_req, d_seq_lens, d_ep_owner, d_ep_page_table, d_tp_page_table,
                    stream);
}

int umm_test_stall_tma_wait(umm_t* u, int32_t layer, uint32_t polls) {
#ifdef UMM_CHECKED
  if (!u || layer < -1 || layer >= u->dims.num_layers) return UMM_ERR_INVALID_ARG;
  u->test_stall_layer = polls ? layer : -1;
  u->test_stall_polls = layer >= 0 ? polls : 0u;
  return UMM_OK;
#else
  (void)u;
  (void)layer;
  (void)polls;
  return UMM_ERR_INVALID_ARG;   // only the checked build carries the hook
#endif
}

int umm_set_switch_overlap(umm_t* u, int32_t enable) {
  if (!u) return UMM_ERR_INVALID_ARG;
  if (enable && !u->side) {
    int dev_now = -1;
    if (cudaGetDevice(&dev_now) != cudaSuccess || dev_now != u->device) return UMM_ERR_INVALID_ARG;
    if (cudaStreamCreateWithFlags(&u->side, cudaStreamNonBlocking) != cudaSuccess ||
        cudaEventCreateWithFlags(&u->ev_fork, cudaEventDisableTiming) != cudaSuccess ||
        cudaEventCreateWithFlags(&u->ev_join, cudaEventDisableTiming) != cudaSuccess) {
      if (u->side) cudaStreamDestroy(u->side);
      if (u->ev_fork) cudaEventDestroy(u->ev_fork);
      u->side = nullptr;
      u->ev_fork = u->ev_join = nullptr;
      return UMM_ERR_CUDA;
    }
  }
  u->overlap = enable != 0;
  return UMM_OK;
}

namespace {

// With overlap on, and both weights (or attention weights) and live KV to
// move, the weight reshards go to the side stream: it first waits for
// `stream` (fork), and `stream` waits for it at the end (join), so the call
// stays one ordered unit on `stream` (and capturable into one graph).
struct SwitchStreams {
  umm* u;
  cudaStream_t main;
  bool forked = false;
  SwitchStreams(umm* uu, void* stream, bool use_side) : u(uu), main(as_stream(stream)) {
    if (use_side && cudaEventRecord(u->ev_fork, main) == cudaSuccess &&
        cudaStreamWaitEvent(u->side, u->ev_fork, 0) == cudaSuccess)
      forked = true;
  }
  void* weights() const { return forked ? static_cast<void*>(u->side) : static_cast<void*>(main); }
  int join() {
    if (!forked) return UMM_OK;
    forked = false;
    if (cudaEventRecord(u->ev_join, u->side) != cudaSuccess || cudaStreamWaitEvent(main, u->ev_join, 0) != cudaSuccess)
      return UMM_ERR_CUDA;
    return UMM_OK;
  }
  ~SwitchStreams() { join(); }
};

}  // namespace

int umm_switch_ep2tp(umm_t* u, int32_t R, int32_t maxp, const int32_t* d_seq_lens, const int32_t* d_ep_owner,
                     const int32_t* d_ep_page_table, const int32_t* d_tp_free_pages, int64_t tp_free_count,
                     int32_t* d_tp_pos, int32_t* d_tp_page_table, void* stream) {
  if (!u) return UMM_ERR_INVALID_ARG;
  const bool w = u->dims.E > 0, a = u->dims.attn_q_heads > 0, kv = u->dims.num_kv_heads > 0;
  // every check that can fail on the host runs before anything is enqueued
  if (w && u->weight_mode != UMM_MODE_EP) return UMM_ERR_MODE;
  if (a && u->attn_mode != UMM_MODE_EP) return UMM_ERR_MODE;
  if (kv) {
    if (u->kv_mode != UMM_MODE_EP) return UMM_ERR_MODE;
    int rc = check_kv_args(u, R, maxp, d_seq_lens, d_ep_owner, d_ep_page_table, d_tp_page_table);
    if (rc) return rc;
    if (R > 0 && (!d_tp_free_pages || !d_tp_pos || tp_free_count < 0)) return UMM_ERR_INVALID_ARG;
  }
  SwitchStreams ss(u, stream, u->overlap && (w || a) && kv && R > 0);
  int rc = UMM_OK;
  if (w && (rc = reshard_weights(u, 1, ss.weights()))) return rc;
  if (a && (rc = reshard_attn(u, 1, ss.weights()))) return rc;
  if (!kv) return UMM_OK;
  if (R > 0) {
    if ((rc = gather_requests_ep2tp(u, R, d_ep_owner, d_tp_pos, stream))) return rc;
    if ((rc = umm_assign_pages(u, 1, R, d_seq_lens, nullptr, d_tp_pos, d_tp_free_pages, tp_free_count,
                               tp_free_count, d_tp_page_table, maxp, stream)))
      return rc;
  }
  if ((rc = reshard_kv(u, 0, R, maxp, d_seq_lens, d_ep_owner, d_ep_page_table, d_tp_page_table, stream,
                       !ss.forked)))
    return rc;
  return ss.join();
}

int umm_switch_tp2ep(umm_t* u, int32_t R, int32_t maxp, const int32_t* d_seq_lens, const int32_t* d_tp_pos,
                     const int32_t* d_tp_page_table, const int32_t* d_ep_free_pages, int64_t ep_free_stride,
                     int64_t ep_free_count, int32_t* d_ep_owner, int32_t* d_local_pos, int32_t* d_ep_page_table,
                     void* stream) {
  if (!u) return UMM_ERR_INVALID_ARG;
  const bool w = u->dims.E > 0, a = u->dims.attn_q_heads > 0, kv = u->dims.num_kv_heads > 0;
  if (w && u->weight_mode != UMM_MODE_TP) return UMM_ERR_MODE;
  if (a && u->attn_mode != UMM_MODE_TP) return UMM_ERR_MODE;
  if (kv) {
    if (u->kv_mode != UMM_MODE_TP) return UMM_ERR_MODE;
    int rc = check_kv_args(u, R, maxp, d_seq_lens, d_ep_owner, d_ep_page_table, d_tp_page_table);
    if (rc) return rc;
    if (R > 0 && (!d_ep_free_pages || !d_local_pos || ep_free_count < 0 ||
                  (u->dims.P > 1 && ep_free_stride < ep_free_count)))
      return UMM_ERR_INVALID_ARG;
  }
  SwitchStreams ss(u, stream, u->overlap && (w || a) && kv && R > 0);
  int rc = UMM_OK;
  auto weights = [&]() {
    if (w && (rc = reshard_weights(u, 0, ss.weights()))) return rc;
    if (a && (rc = reshard_attn(u, 0, ss.weights()))) return rc;
    return UMM_OK;
  };
  if (ss.forked && weights()) return rc;            // beside the bookkeeping below
  if (kv && R > 0) {
    if ((rc = place_requests_tp2ep(u, R, d_seq_lens, d_tp_pos, d_ep_owner, d_local_pos, stream))) return rc;
    if ((rc = umm_assign_pages(u, u->dims.P, R, d_seq_lens, d_ep_owner, d_tp_pos, d_ep_free_pages, ep_free_stride,
                               ep_free_count, d_ep_page_table, maxp, stream)))
      return rc;
  }
  if (!ss.forked && weights()) return rc;
  if (!kv) return UMM_OK;
  if ((rc = reshard_kv(u, 1, R, maxp, d_seq_lens, d_ep_owner, d_ep_page_table, d_tp_page_table, stream))) return rc;
  return ss.join();
}

int umm_kv_check_capacity(const umm_t* u, int32_t target_kv_mode, int32_t R, const int32_t* h_seq_lens,
                          const int32_t* h_ep_owner) {
  if (!u || u->dims.num_kv_heads == 0 || R < 0 || (R > 0 && !h_seq_lens)) return UMM_ERR_INVALID_ARG;
  if (target_kv_mode != UMM_MODE_EP && target_kv_mode != UMM_MODE_TP) return UMM_ERR_INVALID_ARG;
  if (target_kv_mode == UMM_MODE_EP && R > 0 && !h_ep_owner) return UMM_ERR_INVALID_ARG;
  const int64_t ps = u->dims.page_size;
  std::vector<int64_t> per(u->dims.P, 0);
  int64_t total = 0;
  for (int32_t k = 0; k < R; ++k) {
    if (h_seq_lens[k] < 0) return UMM_ERR_BAD_REQUEST;
    const int64_t np = (h_seq_lens[k] + ps - 1) / ps;
    total += np;
    if (target_kv_mode == UMM_MODE_EP) {
      const int32_t o = h_ep_owner[k];
      if (o < 0 || o >= u->dims.P) return UMM_ERR_BAD_REQUEST;
      per[o] += np;
    }
  }
  if (total > u->L.desc_capacity) return UMM_ERR_CAPACITY;
  if (target_kv_mode == UMM_MODE_TP) return total > u->L.pages_tp ? UMM_ERR_CAPACITY : UMM_OK;
  for (int64_t x : per)
    if (x > u->L.pages_ep) return UMM_ERR_CAPACITY;
  return UMM_OK;
}

int umm_status_sync(umm_t* u, void* stream, int32_t* status_out, uint32_t* flags_out) {
  if (!u) return UMM_ERR_INVALID_ARG;
  cudaStream_t s = as_stream(stream);
  umm_status_block blk;
  if (cudaMemcpyAsync(&blk, u->geo.base + u->ws.status, sizeof(blk), cudaMemcpyDeviceToHost, s) != cudaSuccess ||
      cudaStreamSynchronize(s) != cudaSuccess)
    return UMM_ERR_CUDA;
  const uint32_t f = blk.flags;
  int32_t code = UMM_OK;
  if (f & UMM_FLAG_DUP_PAGE) code = UMM_ERR_DUP_PAGE;
  if (f & UMM_FLAG_PAGE_OOB) code = UMM_ERR_PAGE_OOB;
  if (f & UMM_FLAG_CAPACITY) code = UMM_ERR_CAPACITY;
  if (f & UMM_FLAG_BAD_REQUEST) code = UMM_ERR_BAD_REQUEST;
  if (f & UMM_FLAG_TIMEOUT) code = UMM_ERR_TIMEOUT;  // a bounded wait of a TMA copy gave up
  if (f & UMM_FLAG_ACCESS) code = UMM_ERR_ACCESS;    // checked build: a library fault
  if (f & ~(UMM_FLAG_ACCESS | UMM_FLAG_TIMEOUT)) {
    // the first KV reshard at or after the failing call did not run, nor did
    // any later one: the cache is still in the layout that call started from
    for (const KvCall& c : u->kv_log)
      if (c.id >= blk.fail_call) {
        u->kv_mode = c.mode_before;
        break;
      }
  }
  if (f) {
    uint32_t zero[2] = {0, 0};
    if (cudaMemcpyAsync(u->geo.base + u->ws.status, zero, sizeof(zero), cudaMemcpyHostToDevice, s) != cudaSuccess ||
        cudaStreamSynchronize(s) != cudaSuccess)
      return UMM_ERR_CUDA;
  }
  u->kv_log.clear();
  if (status_out) *status_out = code;
  if (flags_out) *flags_out = f;
  return UMM_OK;
}

const char* umm_strerror(int code) {
  switch (code) {
    case UMM_OK: return "ok";
    case UMM_ERR_INVALID_ARG: return "invalid argument";
    case UMM_ERR_ALIGN: return "buffer base not 256-byte aligned";
    case UMM_ERR_MODE: return "data is not in the source layout of this switch";
    case UMM_ERR_CAPACITY: return "target capacity exceeded";
    case UMM_ERR_PAGE_OOB: return "page id out of range";
    case UMM_ERR_CUDA: return "CUDA runtime error";
    case UMM_ERR_TIMEOUT: return "bounded device wait timed out";
    case UMM_ERR_DUP_PAGE: return "destination page used twice";
    case UMM_ERR_BAD_REQUEST: return "bad request metadata (length, owner or list position)";
    case UMM_ERR_ACCESS: return "checked build: an out-of-range or misaligned access was skipped";
    default: return "unknown status";
  }
}

int umm_profile_enable(umm_t* u, int32_t enable) {
  if (!u) return UMM_ERR_INVALID_ARG;
  u->prof = enable != 0;
  if (u->prof && u->ev_pool.empty() && u->pending.empty()) {
    for (int i = 0; i < 8192; ++i) {
      cudaEvent_t e;
      if (cudaEventCreate(&e) != cudaSuccess) return UMM_ERR_CUDA;
      u->ev_pool.push_back(e);
    }
  }
  return UMM_OK;
}

int umm_profile_read(umm_t* u, int32_t kind, int64_t* launches, double* total_ms) {
  if (!u || kind < 0 || kind >= UMM_K_COUNT) return UMM_ERR_INVALID_ARG;
  for (auto& p : u->pending) {
    float ms = 0.f;
    if (cudaEventSynchronize(p.b) != cudaSuccess || cudaEventElapsedTime(&ms, p.a, p.b) != cudaSuccess)
      return UMM_ERR_CUDA;
    u->prof_n[p.kind] += p.units;
    u->prof_ms[p.kind] += ms;
    u->ev_pool.push_back(p.a);
    u->ev_pool.push_back(p.b);
  }
  u->pending.clear();
  if (launches) *launches = u->prof_n[kind];
  if (total_ms) *total_ms = u->prof_ms[kind];
  return UMM_OK;
}

int umm_launch_count(const umm_t* u, int64_t* launches) {
  if (!u || !launches) return UMM_ERR_INVALID_ARG;
  *launches = u->launches;
  return UMM_OK;
}

int umm_profile_reset(umm_t* u) {
  if (!u) return UMM_ERR_INVALID_ARG;
  int64_t n;
  double ms;
  int rc = umm_profile_read(u, 0, &n, &ms);
  if (rc) return rc;
  for (int k = 0; k < UMM_K_COUNT; ++k) {
    u->prof_n[k] = 0;
    u->prof_ms[k] = 0;
  }
  return UMM_OK;
}

}  // extern "C"
