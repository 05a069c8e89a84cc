// Switch policy of the coordinator (host only).
//
// "Moebius: Serving Mixture-of-Expert Models with Seamless Runtime Parallelism
// Switch" (paper review), §4.5: the signal is the global in-flight request
// count, sampled once per decode iteration, after the current step and before
// the next.  The policy is asymmetric:
//  - in TP it moves to EP as soon as the latest count is above T_h;
//  - in EP it moves back to TP only when the mean count of the last W
//    iterations is below T_l (T_l <= T_h gives hysteresis);
//  - after a switch, a cooldown C bounds the switch rate;
//  - before committing, the target layout's KV capacity must hold the live
//    requests; otherwise the switch is cancelled and retried after the
//    cooldown.
// §6.1 gives the evaluation settings: T_h = 256, C = 5 s; interactive serving
// T_l = 0.8 T_h, W = 8; rollout T_l = T_h, W = 1.
#include <new>
#include <vector>

#include "umm.h"

struct umm_policy {
  umm_policy_params p;
  int32_t mode;
  double cool_from;      // time of the last switch or cancellation
  bool cool_active;
  std::vector<int64_t> ring;
  size_t head = 0, filled = 0;
  int64_t sum = 0;
  int64_t switches = 0, cancels = 0;
};

extern "C" {

int umm_policy_create(const umm_policy_params* params, umm_policy_t** out) {
  if (!params || !out) return UMM_ERR_INVALID_ARG;
  const umm_policy_params& p = *params;
  if (p.window < 1 || p.window > (1 << 20) || !(p.t_low <= p.t_high) || !(p.cooldown_s >= 0.0) ||
      (p.start_mode != UMM_MODE_EP && p.start_mode != UMM_MODE_TP))
    return UMM_ERR_INVALID_ARG;
  umm_policy* s = new (std::nothrow) umm_policy();
  if (!s) return UMM_ERR_INVALID_ARG;
  s->p = p;
  s->mode = p.start_mode;
  s->cool_from = 0.0;
  s->cool_active = false;
  s->ring.assign((size_t)p.window, 0);
  *out = s;
  return UMM_OK;
}

int umm_policy_destroy(umm_policy_t* s) {
  if (!s) return UMM_ERR_INVALID_ARG;
  delete s;
  return UMM_OK;
}

int umm_policy_step(umm_policy_t* s, int64_t inflight, double now_s, int32_t target_fits, int32_t* decision) {
  if (!s || !decision || inflight < 0) return UMM_ERR_INVALID_ARG;
  // the window always holds the last W samples, in every mode
  const size_t W = s->ring.size();
  if (s->filled == W) s->sum -= s->ring[s->head];
  else ++s->filled;
  s->ring[s->head] = inflight;
  s->sum += inflight;
  s->head = (s->head + 1) % W;

  *decision = UMM_POLICY_STAY;
  if (s->cool_active && now_s - s->cool_from < s->p.cooldown_s) return UMM_OK;
  bool want = false;
  if (s->mode == UMM_MODE_TP) {
    want = (double)inflight > s->p.t_high;
  } else if (s->filled == W) {
    want = (double)s->sum / (double)W < s->p.t_low;
  }
  if (!want) return UMM_OK;
  s->cool_from = now_s;
  s->cool_active = true;
  if (!target_fits) {
    ++s->cancels;
    *decision = UMM_POLICY_CANCELLED;
    return UMM_OK;
  }
  ++s->switches;
  if (s->mode == UMM_MODE_TP) {
    s->mode = UMM_MODE_EP;
    *decision = UMM_POLICY_TO_EP;
  } else {
    s->mode = UMM_MODE_TP;
    *decision = UMM_POLICY_TO_TP;
  }
  return UMM_OK;
}

int umm_policy_state(const umm_policy_t* s, int32_t* mode, int64_t* switches, int64_t* cancels) {
  if (!s) return UMM_ERR_INVALID_ARG;
  if (mode) *mode = s->mode;
  if (switches) *switches = s->switches;
  if (cancels) *cancels = s->cancels;
  return UMM_OK;
}

}  // extern "C"
