/*
 * umm.h -- C ABI of libumm: the data plane of a runtime EP <-> TP parallelism
 * switch for Mixture-of-Experts serving, on one GPU.
 *
 * Method: "Moebius: Serving Mixture-of-Expert Models with Seamless Runtime
 * Parallelism Switch" (paper review page).  Sections cited below are that
 * paper's:
 *   §3    EP and TP are two layouts of the same bytes; a switch only moves the
 *         bytes whose owner changes.
 *   §3.1  Weight layouts.  EP: rank r owns experts [r*E/P, (r+1)*E/P) whole,
 *         W13 (E/P, 2I, H), W2 (E/P, H, I).  TP: every rank owns a 1/P shard of
 *         every expert, W13 (E, 2I/P, H), W2 (E, H, I/P).
 *   §3.2  KV cache: EP ranks keep all KV heads of their own requests; TP ranks
 *         keep a head shard of every request, heads replicated over rank
 *         groups when KV heads < P.  EP->TP request order comes from a metadata
 *         all-gather; TP->EP placement is greedy (longest first, least-loaded
 *         rank), deterministic.  Paged KV is moved through the page tables.
 *   §4.2, Fig. 7  Unified memory manager: one fixed buffer, N+1 per-layer
 *         slots, TP layer i in slot i and EP layer i in slot i+1; EP->TP walks
 *         layers ascending, TP->EP descending, so the reshard is in place, with
 *         no allocation and fixed tensor addresses (captured graphs stay valid).
 *   §4.3, Table 1, Fig. 8  Fused direct-transfer kernels: one read and one
 *         write per moved element, no staging, page-indexed work descriptors
 *         for the KV cache.
 *   §4.5  Before committing, check that the target layout's KV capacity holds
 *         the live requests.
 *
 * Here the P ranks are P fixed regions of ONE device buffer on one GPU, so
 * every "exchange" is an on-device copy.
 *
 * Conventions for every entry point:
 *  - Return value: UMM_OK (0) or a UMM_ERR_* code.  Host-detectable errors
 *    (bad sizes, null pointers, misalignment, wrong mode) are returned
 *    synchronously and nothing is enqueued.
 *  - Device pointers ("d_" prefix) must point to device memory of the GPU the
 *    buffer lives on; host pointers have the "h_" prefix.  All int32 arrays
 *    are caller-owned; the library never allocates, frees or keeps them.
 *  - `stream` is a cudaStream_t (NULL = legacy default stream).  Calls enqueue
 *    kernels on it and return without synchronising; they call no cudaMalloc
 *    and never move the buffer.  Calls on one handle must be issued to one
 *    stream at a time (they share the workspace).
 *  - Device-detected errors (page table contents, capacity, bad lengths) are
 *    found before any byte of the buffer is written.  They set sticky flags in
 *    the workspace; every later validating kernel (KV, placement, request
 *    order, page hand-out) then does nothing until umm_status_sync() reads and
 *    clears them.  Weight reshards cannot fail on the device and ignore them.
 *  - The per-layer copies of one call (weights, KV, attention) are launched
 *    as a chain: layer k+1 uses programmatic dependent launch, so its CTAs
 *    may start, and read slots that no layer of the call writes, while layer
 *    k drains; each of its stores waits for layer k's grid to complete.
 *    Per-kernel timing (umm_profile_enable) times the chain as a whole, so
 *    it runs chained then too.
 *  - The library never aborts, traps or throws across this ABI.
 *  - A handle is not thread-safe: issue its calls from one host thread, with
 *    the buffer's device current.
 *  - Checked build.  libumm_checked.so is the same library compiled with
 *    UMM_CHECKED: before every vector load or store, the copy kernels (weights,
 *    KV, attention, and the staged variants) test the address against the
 *    buffer it must lie in (the P regions, or the caller's staging buffer) and
 *    against the vector's alignment.  A failing access is skipped and raises
 *    UMM_FLAG_ACCESS (status UMM_ERR_ACCESS).  The checked build serves tests;
 *    the flag can only come from a library fault, never from caller input.
 *    A KV layer already started in the chain when the flag is raised still
 *    runs (it read the flags before the previous layer finished).
 */
#ifndef UMM_H_
#define UMM_H_

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* ---- status codes ---- */
#define UMM_OK               0
#define UMM_ERR_INVALID_ARG  1  /* bad sizes, null pointer, R > max_requests, ...        */
#define UMM_ERR_ALIGN        2  /* buffer base not 256-byte aligned                       */
#define UMM_ERR_MODE         3  /* e.g. EP->TP requested while the data is already TP     */
#define UMM_ERR_CAPACITY     4  /* target pool / descriptor space too small (§4.5)         */
#define UMM_ERR_PAGE_OOB     5  /* a page id outside its pool                             */
#define UMM_ERR_CUDA         6  /* a CUDA runtime call failed (a launch of a multi-kernel
                                   call: the kernels enqueued before it stay enqueued)    */
#define UMM_ERR_TIMEOUT      7  /* a bounded device wait (the mbarrier of a TMA copy) gave
                                   up: that layer copy is incomplete and the KV cache is in
                                   no complete layout (see reshard_kv_ep2tp)              */
#define UMM_ERR_DUP_PAGE     8  /* two live pages would be written to one destination page */
#define UMM_ERR_BAD_REQUEST  9  /* length < 0 or > max_pages_per_req*page_size, owner or
                                   list position out of range                             */
#define UMM_ERR_ACCESS      10  /* checked build only: a kernel formed an address outside
                                   its buffer or off its vector alignment (skipped)       */

#define UMM_MODE_EP 0
#define UMM_MODE_TP 1

/* ---- sizes (§3.1, §3.2) ----
 * P ranks, E experts, H hidden size, I expert intermediate size, num_layers N.
 * Requirements: P >= 1, E % P == 0, I % P == 0, N >= 1.  E == 0 means "no
 * expert weights".  num_kv_heads == 0 means "no KV cache"; otherwise
 * num_kv_heads % P == 0 or P % num_kv_heads == 0, head_dim >= 1,
 * page_size >= 1 and kv_pages_tp a multiple of num_kv_heads / h_tp, where
 * h_tp = max(1, num_kv_heads / P) is the number of heads a TP rank keeps.
 * Elements are 2 bytes (bf16) and are moved as opaque bit patterns. */
typedef struct {
  int32_t P, E, H, I, num_layers;
  int32_t num_kv_heads, head_dim, page_size;
  int64_t kv_pages_tp;     /* TP-view pages per region and KV slot (K and V each)   */
  int32_t max_requests;    /* largest R any request call may pass                   */
  int32_t w13_split;       /* 0: TP rank q keeps gate rows [q*I/P,(q+1)*I/P) then the
                              same rows of up (SwiGLU stays rank-local); 1: rows
                              [q*2I/P, (q+1)*2I/P) of W13                             */
  int64_t max_pages;       /* descriptor capacity: most live pages in one KV call
                              (0 = kv_pages_tp)                                      */
  int32_t weight_mode;     /* layout the weights are in at create (UMM_MODE_*)      */
  int32_t kv_mode;         /* layout the KV cache is in at create                   */
  int32_t attn_q_heads;    /* Hq query heads of the attention weights kept in the
                              memory-saving layout (0 = none); needs
                              num_kv_heads, head_dim, H and Hq % P == 0          */
  int32_t attn_mode;       /* layout the attention weights are in at create       */
} umm_dims;

/* ---- buffer layout (all offsets in bytes from the buffer base) ----
 * region r (rank r) starts at r * region_stride and holds
 *   weight slot s (s = 0..N) at  r*region_stride + s*wslot_stride:
 *       W13 at +w13_off, W2 at +w2_off;
 *       EP view of layer l = slot l+1: W13 [E/P][2I][H], W2 [E/P][H][I]
 *       TP view of layer l = slot l:   W13 [E][2I/P][H], W2 [E][H][I/P]
 *   KV slot s (s = 0..N) at     r*region_stride + kvslots_off + s*kvslot_stride:
 *       K half at +0, V half at +kv_v_off; each half is a page pool
 *       EP view of layer l = slot l+1: [pages_ep][page_size][num_kv_heads][head_dim]
 *       TP view of layer l = slot l:   [pages_tp][page_size][h_tp][head_dim]
 *   attention slot s (s = 0..N) at r*region_stride + attnslots_off + s*attnslot_stride
 *       (only with attn_q_heads > 0): Wqkv at +0, Wo at +attn_wo_off;
 *       EP view of layer l = slot l+1: Wqkv [Hq + 2*Hkv heads][Dh][H], Wo [H][Hq*Dh]
 *       TP view of layer l = slot l:   Wqkv [Hq/P + 2*h_tp heads][Dh][H] (rank q's
 *       query heads, then its key heads, then its value heads), Wo [H][Hq/P*Dh]
 * The workspace (status, descriptors, scratch) follows the P regions at
 * ws_off; callers must not write it.  total_bytes = ws_off + ws_bytes. */
typedef struct {
  uint64_t region_stride, wslot_stride, w13_off, w2_off;
  uint64_t kvslot_stride, kv_v_off, kvslots_off;
  uint64_t ws_off, ws_bytes, total_bytes;
  int64_t pages_ep, pages_tp, h_tp;
  uint64_t status_off;     /* umm_status_block                                      */
  uint64_t desc_off;       /* umm_kv_desc[desc_capacity]                             */
  int64_t desc_capacity;
  uint64_t attnslot_stride, attn_wo_off, attnslots_off;
} umm_layout_t;

/* Workspace status block (device memory, at status_off). */
typedef struct {
  uint32_t flags;          /* sticky UMM_FLAG_* bits                                 */
  uint32_t fail_call;      /* id of the first call that raised a flag (0 = none)     */
  uint64_t ndesc;          /* descriptors written by the last KV call                */
  uint64_t tokens;         /* live tokens of the last KV call                        */
  uint64_t reserved[5];
} umm_status_block;

#define UMM_FLAG_BAD_REQUEST 1u
#define UMM_FLAG_CAPACITY    2u
#define UMM_FLAG_PAGE_OOB    4u
#define UMM_FLAG_DUP_PAGE    8u
#define UMM_FLAG_ACCESS     16u   /* checked build only, see UMM_ERR_ACCESS */
#define UMM_FLAG_TIMEOUT    32u   /* see UMM_ERR_TIMEOUT */

/* One page-indexed work descriptor (§4.3): the live tokens of logical page
 * `page` of request `req`.  Descriptors are grouped by the rank whose bytes
 * they move (EP->TP: the EP owner read from; TP->EP: the EP owner written
 * to), then by request, then by page.  src_region / dst_region = -1 means
 * "per head: the TP rank(s) holding it". */
typedef struct {
  int32_t req, page, src_region, dst_region, src_page, dst_page, ntok, reserved;
} umm_kv_desc;

typedef struct umm umm_t;  /* opaque host handle, owned by the library */

/* Bytes the caller must allocate for `dims` (host-only computation). */
int umm_required_bytes(const umm_dims* dims, uint64_t* bytes_out);

/* Layout for `dims` without a handle (host-only computation). */
int umm_layout_for_dims(const umm_dims* dims, umm_layout_t* out);

/* Bind a handle to a caller-owned device buffer of at least
 * umm_required_bytes() bytes, base 256-byte aligned (§4.2: the one
 * allocation, made once at start-up).  Initialises the workspace's status
 * block and TP-page schedule (synchronous memsets); everything else in the
 * buffer is left as is.
 * Errors: INVALID_ARG, ALIGN, CAPACITY (bytes too small), CUDA. */
int umm_create(const umm_dims* dims, void* d_base, uint64_t bytes, umm_t** out);

/* Release the host handle.  The buffer stays the caller's. */
int umm_destroy(umm_t* u);

int umm_layout(const umm_t* u, umm_layout_t* out);

/* Current layout of the weights and of the KV cache (UMM_MODE_*).  Modes
 * flip when a reshard is enqueued; umm_status_sync() restores the KV mode of
 * a call that a device-detected error stopped. */
int umm_get_modes(const umm_t* u, int32_t* weight_mode, int32_t* kv_mode);

/* Declare which layout the data is in (e.g. after the caller loaded it). */
int umm_set_modes(umm_t* u, int32_t weight_mode, int32_t kv_mode);

/* §3.1, §4.2, §4.3: expert weights EP -> TP, in place, layers ascending (one
 * launch per layer): EP slot l+1 of every region -> TP slot l of every
 * region.  W13 row j = g*I + i of EP expert (r, e_l) goes to TP rank i / (I/P),
 * expert r*E/P + e_l, row g*I/P + i % (I/P) (w13_split 0); W2 column i goes
 * to TP rank i / (I/P), column i % (I/P).  Errors: MODE (weights not in EP),
 * INVALID_ARG (no weights), CUDA. */
int reshard_weights_ep2tp(umm_t* u, void* stream);

/* Inverse of the above, layers descending: TP slot l -> EP slot l+1. */
int reshard_weights_tp2ep(umm_t* u, void* stream);

/* §3.1, memory-saving variant of the attention weights (only the active
 * layout is resident).  EP->TP: every rank keeps its own shard of its full
 * copy (query heads q*Hq/P.., its key and value heads, its Wo columns);
 * nothing crosses ranks.  TP->EP: all-gather -- every rank's full copy is
 * rebuilt from the shards, key/value heads from their lowest replica; each
 * shard element is read once and written to all P ranks.  One launch per
 * layer (ascending / descending, N+1 slots as for the expert weights).
 * Errors: INVALID_ARG (no attention weights), MODE, CUDA. */
int reshard_attn_ep2tp(umm_t* u, void* stream);
int reshard_attn_tp2ep(umm_t* u, void* stream);
int umm_get_attn_mode(const umm_t* u, int32_t* mode);
int umm_set_attn_mode(umm_t* u, int32_t mode);

/* The staged (collective-style) weight reshard, for comparison with the
 * fused one (§4.3, Table 1: a collective path stages per-peer blocks and
 * touches HBM twice; the fused path once).  EP->TP permutes each EP rank's
 * slot into per-peer blocks in `d_stage`, then an exchange copies block
 * (r, q) into TP rank q's slot; TP->EP runs the exchange out of the TP slots,
 * then the permute back into whole experts.  Two reads and two writes per
 * element; same result as the fused calls.  `d_stage`: caller-owned device
 * memory, 256-byte aligned, at least umm_weights_stage_bytes() bytes
 * (P*P blocks, one layer).  Errors as the fused calls, plus ALIGN and
 * CAPACITY (staging too small). */
int umm_weights_stage_bytes(const umm_t* u, uint64_t* bytes_out);
int reshard_weights_ep2tp_staged(umm_t* u, void* d_stage, uint64_t stage_bytes, void* stream);
int reshard_weights_tp2ep_staged(umm_t* u, void* d_stage, uint64_t stage_bytes, void* stream);

/* §3.2 EP -> TP request order (metadata all-gather): the global list is rank
 * 0's requests, then rank 1's, ..., each rank's in ascending request index.
 * d_tp_pos[k] receives request k's position.  d_ep_owner[k] in [0, P).
 * Device errors: BAD_REQUEST (owner out of range; d_tp_pos untouched). */
int gather_requests_ep2tp(umm_t* u, int32_t R, const int32_t* d_ep_owner, int32_t* d_tp_pos,
                          void* stream);

/* §3.2 TP -> EP placement: requests sorted by length descending (ties: list
 * position ascending), each to the rank with the least load so far (load =
 * tokens; ties: lowest rank).  d_list_pos[k] = request k's position in the
 * global list (a permutation of 0..R-1), or NULL for "position = k".
 * Outputs d_owner[k] and d_local_pos[k] (rank of k among its owner's requests
 * by list position).  Device errors: BAD_REQUEST (negative length or list
 * positions not a permutation; outputs untouched). */
int place_requests_tp2ep(umm_t* u, int32_t R, const int32_t* d_seq_lens, const int32_t* d_list_pos,
                         int32_t* d_owner, int32_t* d_local_pos, void* stream);

/* The placement above, for callers that cannot allocate device memory.
 * (The paper has no counterpart: this entry point exists for deployments.)
 * place_requests_tp2ep() needs a handle, and the handle needs a unified
 * buffer that someone cudaMalloc'ed.  A scheduler process that only receives
 * device pointers to request metadata, or code running where an allocator must
 * not be entered (inside allocator callbacks, under a strict memory budget,
 * while other work is being captured), cannot provide one.  This variant takes
 * no handle and allocates nothing: its scratch (the list-position -> request
 * map and the rank chosen per sorted position) is two fixed arrays of this
 * library's own device memory, 80 KiB together, which a GPU keeps from this
 * entry point's first call on it until the process exits.
 *  - P in [1, 64]; R in [0, 16384]: a larger R is refused with
 *    UMM_ERR_CAPACITY before anything is enqueued.
 *  - Same arguments and results as place_requests_tp2ep(); d_status (device
 *    int32, may be NULL) receives UMM_OK or UMM_ERR_BAD_REQUEST (negative
 *    length, or list positions that are not a permutation; outputs are then
 *    untouched).  With R == 0 nothing is enqueued and d_status is not written.
 *  - All calls on one GPU share the scratch array: calls whose kernels may
 *    overlap on the GPU (unordered streams) race; order them on one stream.
 *  - The first call on each device (R == 0 included) does the set-up: it
 *    looks up the arrays' addresses and sets the kernel's shared-memory
 *    limit.  Under CUDA's lazy module loading (the default), this is when the
 *    driver loads the entry point's device code and arrays onto the device,
 *    which may take device memory.  Make that first call at start-up, before
 *    any stream capture; later calls take no device memory. */
int place_requests_tp2ep_noalloc(int32_t P, int32_t R, const int32_t* d_seq_lens, const int32_t* d_list_pos,
                                 int32_t* d_owner, int32_t* d_local_pos, int32_t* d_status, void* stream);

/* Destination pages for a switch, handed out from free lists in list order
 * (the page's "reassigned target pages", §3.2).  Pool g's free pages are
 * d_free_pages[g*free_stride + 0 .. free_count-1]; request k draws from pool
 * d_pool[k] (NULL = pool 0) and requests of a pool are served in ascending
 * d_key order (NULL = request index; keys must be a permutation of 0..R-1),
 * each taking ceil(len/page_size) consecutive free entries.  Writes
 * d_page_table[k*max_pages_per_req + p], -1 past the request's pages.
 * Device errors: CAPACITY (a pool runs out), BAD_REQUEST (bad length, pool or
 * key); on error the table is untouched. */
int umm_assign_pages(umm_t* u, int32_t npools, int32_t R, const int32_t* d_seq_lens,
                     const int32_t* d_pool, const int32_t* d_key, const int32_t* d_free_pages,
                     int64_t free_stride, int64_t free_count, int32_t* d_page_table,
                     int32_t max_pages_per_req, void* stream);

/* §3.2, §4.3, Fig. 8b: paged KV EP -> TP, in place, layers ascending.
 * Request k (length d_seq_lens[k]) is owned by EP rank d_ep_owner[k]; its
 * logical page p sits at EP page d_ep_page_table[k*maxp + p] of that rank
 * and goes to TP page d_tp_page_table[k*maxp + p] on every rank holding each
 * head (TP page ids are the same on all ranks).  Token t of page p is row
 * t % page_size.  One descriptor-building pass (validation first), then one
 * gather/scatter launch per layer; each source row is read once and stored to
 * every replica.  Bytes of pages past a request's length, and of unused
 * pages, are not written.  When every TP rank holds one head (num_kv_heads
 * <= P) and a head row is a multiple of 16 bytes, the copy runs through TMA:
 * tensor-map loads de-interleave each head of an EP page into shared memory
 * and bulk stores write its live rows to each replica.  Errors: MODE,
 * INVALID_ARG (sync); BAD_REQUEST, CAPACITY, PAGE_OOB, DUP_PAGE (device,
 * before any write); TIMEOUT (the TMA copy's bounded wait gave up; not
 * expected).  After TIMEOUT: the layers before the one whose wait ran out
 * were copied; a CTA whose wait ran out stored nothing, other CTAs of that
 * layer may have stored their pages; the next layer may have copied pages
 * too if it had started under programmatic dependent launch before the flag
 * was raised; later layers stored nothing.  The handle stays usable
 * (umm_status_sync() clears the flag), but the KV cache must be rebuilt or
 * reloaded by the caller, who then declares its layout with umm_set_modes().
 * A CTA waits for its own loads at most twice (each a bounded number of
 * polls) before it leaves; should both run out, a load may still write that
 * CTA's shared memory after it has exited.  Tensor-map coordinates are
 * {element, head, row in page, page, region}, each below 2^31 for every
 * accepted pool size. */
int reshard_kv_ep2tp(umm_t* u, int32_t R, int32_t max_pages_per_req, const int32_t* d_seq_lens,
                     const int32_t* d_ep_owner, const int32_t* d_ep_page_table,
                     const int32_t* d_tp_page_table, void* stream);

/* Paged KV TP -> EP, layers descending: request k goes to its new EP owner
 * d_ep_owner[k] (from place_requests_tp2ep), logical page p from TP page
 * d_tp_page_table[k*maxp+p] to EP page d_ep_page_table[k*maxp+p] of that
 * owner; each head is read from the lowest TP rank holding it. */
int reshard_kv_tp2ep(umm_t* u, int32_t R, int32_t max_pages_per_req, const int32_t* d_seq_lens,
                     const int32_t* d_ep_owner, const int32_t* d_ep_page_table,
                     const int32_t* d_tp_page_table, void* stream);

/* Which copy kernel a KV reshard of `dims` launches per layer (host-only;
 * no GPU needed).  The paper has no counterpart: this reports an
 * implementation choice of this library (§3.2 and §4.3 fix only what moves).  dir 0 = EP->TP, 1 = TP->EP.  *kernel = UMM_KV_COPY_TMA
 * (EP->TP through tensor-map loads and bulk stores, see reshard_kv_ep2tp) or
 * UMM_KV_COPY_LSU (vector loads and stores with 64-bit offsets);
 * *vector_bytes (may be NULL) receives the LSU copy's vector width, 0 for
 * TMA.  This is the shape's choice: reshard_kv_ep2tp still runs the LSU copy
 * when the driver cannot encode the tensor map, and so does a one-call
 * switch whose weight copies run on the side stream (umm_set_switch_overlap).
 * Errors: INVALID_ARG (bad dims, no KV cache, bad dir, kernel NULL). */
#define UMM_KV_COPY_LSU 0
#define UMM_KV_COPY_TMA 1
int umm_kv_copy_kernel(const umm_dims* dims, int32_t dir, int32_t* kernel, int32_t* vector_bytes);

/* Test hook of the checked build (libumm_checked.so; libumm.so returns
 * UMM_ERR_INVALID_ARG and does nothing).  The paper has no counterpart: it
 * exercises this library's bounded device wait.  From the next KV EP->TP call of
 * this handle on, every CTA of the TMA copy of layer `layer` makes, once its
 * tensor loads have landed, one more wait on a barrier that never completes,
 * limited to `polls` polls.  That wait runs out and the CTA takes the exit of
 * a timed-out wait with no copy in flight: it raises UMM_FLAG_TIMEOUT and
 * stores nothing.  Kernels enqueued after the call see the flag and do
 * nothing until umm_status_sync() reports UMM_ERR_TIMEOUT.  With `layer` the
 * call's last layer, exactly the earlier layers are copied (see
 * reshard_kv_ep2tp for a layer in the middle).  layer = -1 or polls = 0
 * turns it off.
 * Errors: INVALID_ARG (layer outside [-1, num_layers), or libumm.so). */
int umm_test_stall_tma_wait(umm_t* u, int32_t layer, uint32_t polls);

/* The staged (collective-style) KV reshard, for comparison with the fused
 * one (§3.2: gather scattered token slots into per-peer contiguous blocks,
 * exchange them once, scatter into the target pages; §4.3, Table 1).  Same
 * arguments and result as the fused calls; each layer moves one EP rank at a
 * time through `d_stage` (caller-owned device memory, 256-byte aligned, at
 * least umm_kv_stage_bytes(): a send and a receive area for one rank's live
 * tokens at full EP capacity).  Every replicated row crosses HBM three times
 * (gather, exchange, scatter) instead of once.  Errors as the fused calls,
 * plus ALIGN and CAPACITY (staging too small). */
int umm_kv_stage_bytes(const umm_t* u, uint64_t* bytes_out);
int reshard_kv_ep2tp_staged(umm_t* u, void* d_stage, uint64_t stage_bytes, int32_t R, int32_t max_pages_per_req,
                            const int32_t* d_seq_lens, const int32_t* d_ep_owner, const int32_t* d_ep_page_table,
                            const int32_t* d_tp_page_table, void* stream);
int reshard_kv_tp2ep_staged(umm_t* u, void* d_stage, uint64_t stage_bytes, int32_t R, int32_t max_pages_per_req,
                            const int32_t* d_seq_lens, const int32_t* d_ep_owner, const int32_t* d_ep_page_table,
                            const int32_t* d_tp_page_table, void* stream);

/* One whole switch, one call per direction (the "switch between decode
 * steps" of §3.2 / §4.1): the expert weights (when E > 0), the attention
 * weights (when attn_q_heads > 0) and, when the KV cache exists, the request
 * bookkeeping and the KV reshard, all enqueued on `stream` in this order.
 *
 * umm_switch_ep2tp: weights, attention, gather_requests_ep2tp (-> d_tp_pos),
 *   TP pages from d_tp_free_pages in list order (umm_assign_pages, one pool
 *   -> d_tp_page_table), reshard_kv_ep2tp.
 * umm_switch_tp2ep: place_requests_tp2ep (list positions d_tp_pos ->
 *   d_ep_owner, d_local_pos), EP pages from each owner's free list
 *   (d_ep_free_pages[g*ep_free_stride ..] -> d_ep_page_table), weights,
 *   attention, reshard_kv_tp2ep.
 * Host-detectable errors (modes, arguments) are found before anything is
 * enqueued; device-detected ones follow umm_status_sync(). */
int umm_switch_ep2tp(umm_t* u, int32_t R, int32_t max_pages_per_req, const int32_t* d_seq_lens,
                     const int32_t* d_ep_owner, const int32_t* d_ep_page_table, const int32_t* d_tp_free_pages,
                     int64_t tp_free_count, int32_t* d_tp_pos, int32_t* d_tp_page_table, void* stream);
int umm_switch_tp2ep(umm_t* u, int32_t R, int32_t max_pages_per_req, const int32_t* d_seq_lens,
                     const int32_t* d_tp_pos, const int32_t* d_tp_page_table, const int32_t* d_ep_free_pages,
                     int64_t ep_free_stride, int64_t ep_free_count, int32_t* d_ep_owner, int32_t* d_local_pos,
                     int32_t* d_ep_page_table, void* stream);

/* Opt-in (default off): in umm_switch_ep2tp / umm_switch_tp2ep the weight
 * and attention-weight reshards run on a side stream of the handle, beside
 * the request bookkeeping and the KV reshard on `stream`.  They touch
 * disjoint slots, so the result is the same; the side stream waits for
 * `stream` at the start of the call and `stream` waits for it at the end, so
 * a call stays one ordered unit on `stream` (and one unit in a captured
 * graph).  It shortens switches with little KV to move, where the fixed
 * weight copy dominates.  Per-kernel times read through umm_profile_* then
 * overlap.  The first enable creates the side stream and two events: make it
 * with the buffer's device current, before any stream capture.  Applies only
 * when the call has both weights (or attention weights) and live KV.
 * Errors: INVALID_ARG (null handle, other device current), CUDA. */
int umm_set_switch_overlap(umm_t* u, int32_t enable);

/* §4.5 capacity check on the host, before committing a switch: UMM_OK if the
 * target layout's KV pools hold the requests (TP: all pages in one pool of
 * pages_tp; EP: each owner's pages within pages_ep), else UMM_ERR_CAPACITY.
 * h_ep_owner is needed for target UMM_MODE_EP only. */
int umm_kv_check_capacity(const umm_t* u, int32_t target_kv_mode, int32_t R,
                          const int32_t* h_seq_lens, const int32_t* h_ep_owner);

/* Synchronise `stream`, read the sticky device flags, clear them, and return
 * the highest-priority code among them (ACCESS > TIMEOUT > BAD_REQUEST >
 * CAPACITY > PAGE_OOB > DUP_PAGE; UMM_OK if none) in *status_out (flags in
 * *flags_out, may be NULL).  If a KV reshard was stopped by a validation
 * flag, the handle's KV mode is set back to the layout the data is actually
 * in; ACCESS and TIMEOUT leave it (that reshard ran, with copies missing: see
 * reshard_kv_ep2tp for what TIMEOUT leaves behind). */
int umm_status_sync(umm_t* u, void* stream, int32_t* status_out, uint32_t* flags_out);

/* Static description of a status code. */
const char* umm_strerror(int code);

/* Per-kernel timing with CUDA events recorded on the launching stream
 * (diagnostics; not for use under graph capture).  The layer copies of one
 * call (weights, KV, attention; fused or staged) are timed by one event pair
 * around all of them, so their launch chain stays intact, and count one unit
 * per layer; the descriptor pass, placement, order and page hand-out count
 * one unit per call.  Kinds: */
#define UMM_K_WEIGHTS_EP2TP 0
#define UMM_K_WEIGHTS_TP2EP 1
#define UMM_K_KV_PREP       2
#define UMM_K_KV_EP2TP      3
#define UMM_K_KV_TP2EP      4
#define UMM_K_PLACE         5
#define UMM_K_ORDER         6
#define UMM_K_ASSIGN        7
#define UMM_K_ATTN_EP2TP    8
#define UMM_K_ATTN_TP2EP    9
#define UMM_K_COUNT         10
int umm_profile_enable(umm_t* u, int32_t enable);
/* Synchronises the recorded events; units (see above) and summed
 * milliseconds of one kind since the last reset: total_ms / units is the
 * average time of one layer copy (or one call). */
int umm_profile_read(umm_t* u, int32_t kind, int64_t* launches, double* total_ms);
int umm_profile_reset(umm_t* u);

/* Number of kernels this handle has enqueued since umm_create (counted on
 * the host at launch time). */
int umm_launch_count(const umm_t* u, int64_t* launches);

/* ---- switch policy (host only; §4.5, settings of §6.1) ----
 * Decides, once per decode iteration, whether to switch layouts:
 *  - in TP, switch to EP as soon as the latest in-flight count > t_high;
 *  - in EP, switch to TP only when the mean of the last `window` counts is
 *    < t_low (t_low <= t_high: hysteresis); the window holds the last
 *    `window` samples in every mode and must be full;
 *  - no decision for cooldown_s seconds after a switch or a cancellation;
 *  - a wanted switch whose target layout cannot hold the live requests
 *    (target_fits = 0, e.g. from umm_kv_check_capacity) is cancelled and
 *    retried after the cooldown.
 * Deterministic: the same inputs give the same decisions. */
typedef struct {
  double t_high, t_low;    /* thresholds on the in-flight request count       */
  int32_t window;          /* W >= 1 iterations averaged in EP                 */
  double cooldown_s;       /* C >= 0 seconds                                    */
  int32_t start_mode;      /* UMM_MODE_EP or UMM_MODE_TP                        */
} umm_policy_params;

#define UMM_POLICY_STAY      0
#define UMM_POLICY_TO_EP     1
#define UMM_POLICY_TO_TP     2
#define UMM_POLICY_CANCELLED 3

typedef struct umm_policy umm_policy_t;
int umm_policy_create(const umm_policy_params* params, umm_policy_t** out);
int umm_policy_destroy(umm_policy_t* policy);
/* One iteration: in-flight count after the step that just finished, the time
 * (seconds, non-decreasing) and whether the layout a switch would go to holds
 * the live requests.  *decision = UMM_POLICY_*; the policy's mode follows
 * UMM_POLICY_TO_EP / UMM_POLICY_TO_TP. */
int umm_policy_step(umm_policy_t* policy, int64_t inflight, double now_s, int32_t target_fits,
                    int32_t* decision);
int umm_policy_state(const umm_policy_t* policy, int32_t* mode, int64_t* switches, int64_t* cancels);

#ifdef __cplusplus
}
#endif

#endif /* UMM_H_ */
