"""Named synthetic workloads (sizes, seeds and request-length mixes).

Shapes follow the weight layouts of §3.1 and the paged KV of §3.2 of
"Moebius: Serving Mixture-of-Expert Models with Seamless Runtime Parallelism
Switch"; the model and traces of that page are not available, so these seeded
synthetic stand-ins are used instead.  No reshard arithmetic lives here.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, replace

import numpy as np

from . import RAW, NORMAL, lengths_lognormal, lengths_uniform, npages


@dataclass(frozen=True)
class Workload:
    name: str
    P: int
    N: int
    E: int = 0
    H: int = 0
    I: int = 0
    Hkv: int = 0
    D: int = 0
    ps: int = 16
    R: int = 0
    len_kind: str = "uniform"      # "uniform" (lo..hi) or "lognormal" (median, sigma, cap)
    len_a: float = 1
    len_b: float = 1
    len_cap: int = 1
    w_sigma: float | None = None   # None = raw 16-bit patterns
    kv_sigma: float | None = None
    seed: int = 0
    slack: float = 1.02            # TP page pool = slack * pages in use
    Hq: int = 0                    # attention query heads (0 = no attention weights)

    @property
    def h_tp(self) -> int:
        return self.Hkv // self.P if self.Hkv >= self.P else 1

    def lengths(self) -> np.ndarray:
        if self.R == 0 or self.Hkv == 0:
            return np.zeros(0, dtype=np.int32)
        if self.len_kind == "uniform":
            return lengths_uniform(self.seed, self.R, int(self.len_a), int(self.len_b))
        return lengths_lognormal(self.seed, self.R, self.len_a, self.len_b, self.len_cap)

    def max_pages_per_req(self) -> int:
        cap = int(self.len_b) if self.len_kind == "uniform" else self.len_cap
        return max(1, (cap + self.ps - 1) // self.ps)

    def pages_tp(self) -> int:
        """TP page pool per region and KV slot: slack over the pages in use,
        rounded up so that the EP view (all heads per page) has whole pages."""
        if self.Hkv == 0:
            return 0
        if self.R == 0:       # heads without a cache (attention weights only)
            return self.Hkv // self.h_tp
        used = int(npages(self.lengths(), self.ps).sum())
        n = max(1, math.ceil(self.slack * used))
        m = self.Hkv // self.h_tp
        return (n + m - 1) // m * m

    def dims(self) -> dict:
        ptp = self.pages_tp()
        return dict(P=self.P, E=self.E, H=self.H, I=self.I, N=self.N, Hkv=self.Hkv, D=self.D,
                    ps=self.ps, pages_tp=ptp, max_requests=max(self.R, 1),
                    max_pages=max(ptp, 1), w13_split=0, Hq=self.Hq)

    def w_mode(self):
        return (RAW, 1.0) if self.w_sigma is None else (NORMAL, self.w_sigma)

    def kv_mode(self):
        return (RAW, 1.0) if self.kv_sigma is None else (NORMAL, self.kv_sigma)

    def with_(self, **kw) -> "Workload":
        return replace(self, **kw)


# The five workloads of the build's scope, by what they are.
TINY = Workload("tiny_p2_e8_h64_i32_kv4req", P=2, N=2, E=8, H=64, I=32, Hkv=2, D=16, ps=16,
                R=4, len_kind="uniform", len_a=1, len_b=40)
WEIGHTS_H2048 = Workload("weights_p8_e128_h2048_i768_4layers", P=8, N=4, E=128, H=2048, I=768,
                         w_sigma=0.02)
WEIGHTS_H4096 = Workload("weights_p8_e128_h4096_i1536_8layers", P=8, N=8, E=128, H=4096, I=1536,
                         w_sigma=0.02)
KV_256REQ = Workload("kv_p8_8layers_256req_u1k-32k_hkv4_d128", P=8, N=8, Hkv=4, D=128, ps=16,
                     R=256, len_kind="uniform", len_a=1024, len_b=32768, kv_sigma=1.0)
FULL_SWITCH = Workload("full_switch_p8_e128_h2048_i768_8layers_2048req_lognormal_hkv4_d128",
                       P=8, N=8, E=128, H=2048, I=768, Hkv=4, D=128, ps=16, R=2048,
                       len_kind="lognormal", len_a=2048, len_b=1.0, len_cap=32768,
                       w_sigma=0.02, kv_sigma=1.0)

# Small cases of the same kernels for ncu captures (a few GB on the device,
# per-launch traffic still far above the 129 MB L2).
KV_PROFILE = KV_256REQ.with_(name="kv_p8_2layers_8req_u1k-32k_hkv4_d128", N=2, R=8)
WEIGHTS_PROFILE = WEIGHTS_H2048.with_(name="weights_p8_e128_h2048_i768_2layers", N=2)

# Attention weights of the page's model shape (64 query / 4 KV heads of 128,
# hidden 4096), memory-saving variant, 8 layers.
ATTN_QWEN3_SHAPE = Workload("attn_p8_h4096_hq64_hkv4_d128_8layers", P=8, N=8, H=4096, Hkv=4, D=128, Hq=64,
                            w_sigma=0.02)

# Small cases for ncu captures of the attention kernel (one layer of the shape
# above, 2.3 GB on the device) and of the request-metadata kernels (placement,
# page hand-out, descriptor pass: 2048 requests of 1..64 tokens, one layer).
ATTN_PROFILE = ATTN_QWEN3_SHAPE.with_(name="attn_p8_h4096_hq64_hkv4_d128_1layer", N=1)
META_PROFILE = Workload("meta_p8_1layer_2048req_u1-64_hkv4_d128", P=8, N=1, Hkv=4, D=128, ps=16, R=2048,
                        len_kind="uniform", len_a=1, len_b=64, kv_sigma=1.0)

ALL = {w.name: w for w in (TINY, WEIGHTS_H2048, WEIGHTS_H4096, KV_256REQ, FULL_SWITCH, KV_PROFILE,
                           WEIGHTS_PROFILE, ATTN_QWEN3_SHAPE, ATTN_PROFILE, META_PROFILE)}
