/*
 * The C ABI used from plain C (C99): this file includes umm.h, links
 * libumm.so and calls the entry points that need no GPU -- layout sizing,
 * host argument checks, status strings and the switch policy -- then prints
 * what it got, one "key value" pair per line, for the test that compares it
 * with the Python binding (tests/test_abi_host.py).  Every other entry point
 * is referenced too, so a declaration that C cannot compile or link fails here.
 */
#include <stdint.h>
#include <stdio.h>
#include <string.h>

#include "umm.h"

typedef void (*any_fn)(void);

int main(void) {
  /* every declared entry point must link */
  const any_fn fns[] = {
      (any_fn)umm_required_bytes, (any_fn)umm_layout_for_dims, (any_fn)umm_create, (any_fn)umm_destroy,
      (any_fn)umm_layout, (any_fn)umm_get_modes, (any_fn)umm_set_modes, (any_fn)reshard_weights_ep2tp,
      (any_fn)reshard_weights_tp2ep, (any_fn)gather_requests_ep2tp, (any_fn)place_requests_tp2ep,
      (any_fn)place_requests_tp2ep_noalloc, (any_fn)umm_assign_pages, (any_fn)reshard_kv_ep2tp,
      (any_fn)reshard_kv_tp2ep, (any_fn)umm_kv_check_capacity, (any_fn)umm_status_sync, (any_fn)umm_strerror,
      (any_fn)umm_profile_enable, (any_fn)umm_profile_read, (any_fn)umm_profile_reset,
      (any_fn)umm_launch_count, (any_fn)umm_weights_stage_bytes, (any_fn)reshard_weights_ep2tp_staged,
      (any_fn)reshard_weights_tp2ep_staged, (any_fn)umm_kv_stage_bytes, (any_fn)reshard_kv_ep2tp_staged,
      (any_fn)reshard_kv_tp2ep_staged, (any_fn)reshard_attn_ep2tp, (any_fn)reshard_attn_tp2ep,
      (any_fn)umm_get_attn_mode, (any_fn)umm_set_attn_mode, (any_fn)umm_switch_ep2tp,
      (any_fn)umm_switch_tp2ep, (any_fn)umm_policy_create, (any_fn)umm_policy_destroy,
      (any_fn)umm_policy_step, (any_fn)umm_policy_state, (any_fn)umm_set_switch_overlap,
      (any_fn)umm_kv_copy_kernel, (any_fn)umm_test_stall_tma_wait};
  for (size_t i = 0; i < sizeof(fns) / sizeof(fns[0]); ++i)
    if (!fns[i]) return 10;
  printf("entry_points %zu\n", sizeof(fns) / sizeof(fns[0]));
  printf("sizeof_dims %zu\nsizeof_layout %zu\nsizeof_status %zu\nsizeof_desc %zu\n", sizeof(umm_dims),
         sizeof(umm_layout_t), sizeof(umm_status_block), sizeof(umm_kv_desc));

  /* the full-switch shape: 8 ranks, 128 experts, H 2048, I 768, 8 layers,
     4 KV heads of 128, page 16, 441,304 TP pages, 2048 requests */
  umm_dims d;
  memset(&d, 0, sizeof(d));
  d.P = 8; d.E = 128; d.H = 2048; d.I = 768; d.num_layers = 8;
  d.num_kv_heads = 4; d.head_dim = 128; d.page_size = 16; d.kv_pages_tp = 441304;
  d.max_requests = 2048; d.max_pages = 441304;
  uint64_t bytes = 0;
  if (umm_required_bytes(&d, &bytes) != UMM_OK) return 11;
  umm_layout_t L;
  if (umm_layout_for_dims(&d, &L) != UMM_OK) return 12;
  printf("required_bytes %llu\n", (unsigned long long)bytes);
  printf("region_stride %llu\nwslot_stride %llu\nkvslot_stride %llu\nkvslots_off %llu\nws_off %llu\n",
         (unsigned long long)L.region_stride, (unsigned long long)L.wslot_stride,
         (unsigned long long)L.kvslot_stride, (unsigned long long)L.kvslots_off, (unsigned long long)L.ws_off);
  printf("pages_ep %lld\nh_tp %lld\n", (long long)L.pages_ep, (long long)L.h_tp);

  /* host-side argument checks return codes and enqueue nothing */
  umm_dims bad = d;
  bad.E = 127;                                   /* E % P != 0 */
  printf("bad_experts %d\n", umm_required_bytes(&bad, &bytes));
  bad = d;
  bad.num_kv_heads = 3;                          /* neither divides the other */
  printf("bad_heads %d\n", umm_required_bytes(&bad, &bytes));
  printf("null_handle %d\n", reshard_weights_ep2tp(NULL, NULL));
  printf("strerror_capacity %s\n", umm_strerror(UMM_ERR_CAPACITY));
  int32_t kern = -1, vbytes = -1;
  printf("kv_copy_ep2tp_rc %d\n", umm_kv_copy_kernel(&d, 0, &kern, &vbytes));
  printf("kv_copy_ep2tp %d %d\n", kern, vbytes);
  printf("kv_copy_tp2ep_rc %d\n", umm_kv_copy_kernel(&d, 1, &kern, &vbytes));
  printf("kv_copy_tp2ep %d %d\n", kern, vbytes);
  printf("stall_hook_null %d\n", umm_test_stall_tma_wait(NULL, 0, 1));

  /* the switch policy (host C++): a burst above T_h switches to EP */
  umm_policy_params pp;
  pp.t_high = 256.0; pp.t_low = 204.8; pp.window = 8; pp.cooldown_s = 5.0; pp.start_mode = UMM_MODE_TP;
  umm_policy_t* pol = NULL;
  if (umm_policy_create(&pp, &pol) != UMM_OK) return 13;
  const int64_t counts[] = {100, 200, 300};
  int32_t decision = -1, mode = -1;
  for (int t = 0; t < 3; ++t)
    if (umm_policy_step(pol, counts[t], (double)t, 1, &decision) != UMM_OK) return 14;
  int64_t switches = 0, cancels = 0;
  umm_policy_state(pol, &mode, &switches, &cancels);
  printf("policy_last_decision %d\npolicy_mode %d\npolicy_switches %lld\n", decision, mode, (long long)switches);
  umm_policy_destroy(pol);
  return 0;
}
