"""GPU-side test scaffolding: a unified buffer from torch, bound to a libumm
handle, filled by the synth generator, plus host copies for the oracle."""
from __future__ import annotations

import numpy as np
import torch

import ep_tp_weight_gb300 as umm
import synth
from helpers import dims_of, fill_plan
from synth.workloads import Workload

_tables: dict[float, torch.Tensor] = {}

# Guard bands before and after every test buffer, filled with patterns that
# close() checks: a kernel that writes outside the unified buffer fails the test.
GUARD = 64 << 10
GUARD_LO, GUARD_HI = 0xA5, 0x5A


def table_dev(sigma: float) -> torch.Tensor:
    if sigma not in _tables:
        _tables[sigma] = torch.from_numpy(synth.normal_table(sigma).view(np.int16).copy()).cuda()
    return _tables[sigma]


def lib_dims(w: Workload, **over):
    d = w.dims()
    d.update(over)
    return umm.make_dims(P=d["P"], E=d["E"], H=d["H"], I=d["I"], N=d["N"], Hkv=d["Hkv"], D=d["D"],
                         ps=d["ps"], pages_tp=d["pages_tp"], max_requests=d["max_requests"],
                         max_pages=d["max_pages"], w13_split=d["w13_split"],
                         weight_mode=d.get("weight_mode", umm.UMM_MODE_EP),
                         kv_mode=d.get("kv_mode", umm.UMM_MODE_EP), Hq=d.get("Hq", 0))


def fill_device(buf: torch.Tensor, L: dict, w: Workload, seed: int, stream=None) -> None:
    base = buf.data_ptr()
    s = 0 if stream is None else stream.cuda_stream
    for a, n, mode, sigma in fill_plan(L, w):
        synth.fill_device(base + 2 * a, n, seed, mode, table_dev(sigma).data_ptr() if mode else 0,
                          base=a, stream=s)


class DevUMM:
    """A caller-owned device buffer (one torch allocation) and its handle."""

    def __init__(self, w: Workload, seed: int = 0, fill: bool = True, **over):
        self.w = w
        self.seed = seed
        self.d = dims_of(w, **{k: v for k, v in over.items() if k not in ("weight_mode", "kv_mode")})
        self.dims = lib_dims(w, **over)
        self.nbytes = umm.umm_required_bytes(self.dims)
        self.raw = torch.empty(self.nbytes + 2 * GUARD, dtype=torch.uint8, device="cuda")
        self.raw[:GUARD].fill_(GUARD_LO)
        self.raw[GUARD + self.nbytes:].fill_(GUARD_HI)
        self.buf = self.raw[GUARD:GUARD + self.nbytes]
        self.h = umm.umm_create(self.dims, self.buf, self.nbytes)
        self.L = umm.umm_layout(self.h)
        if fill:
            fill_device(self.buf, self.L, w, seed)
            torch.cuda.synchronize()

    def host(self) -> np.ndarray:
        torch.cuda.synchronize()
        return self.buf[:self.L["ws_off"]].cpu().numpy()

    def u16(self) -> torch.Tensor:
        return self.buf[:self.L["ws_off"]].view(torch.int16)

    def status(self):
        return umm.umm_status_sync(self.h)

    def guards_intact(self) -> bool:
        torch.cuda.synchronize()
        return bool((self.raw[:GUARD] == GUARD_LO).all().item() and
                    (self.raw[GUARD + self.nbytes:] == GUARD_HI).all().item())

    def close(self) -> None:
        if self.h:
            umm.umm_destroy(self.h)
            self.h = None
        intact = self.raw is None or self.guards_intact()
        self.buf = None
        self.raw = None
        torch.cuda.empty_cache()
        assert intact, "a kernel wrote into the guard bands around the unified buffer"


def i32(a) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(np.asarray(a, dtype=np.int32))).cuda()
