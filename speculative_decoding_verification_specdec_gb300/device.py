"""Device-side marshalling: copy a host batch to CUDA tensors, allocate the outputs, call
the library. No arithmetic of the method happens here."""
from __future__ import annotations

import dataclasses
from typing import Dict, Optional

import numpy as np

from . import _native
from .workloads import BF16, Workload

INPUT_FIELDS = ("logits", "draft_ids", "draft_probs", "has_q", "cu_num_draft", "bitmask", "temperature",
                "uniforms", "exp_noise", "top_k", "top_p")


def _host_tensor(a: np.ndarray, bf16: bool = False):
    import torch

    t = torch.from_numpy(np.ascontiguousarray(a))
    if bf16:
        t = t.view(torch.int16).view(torch.bfloat16)
    return t


def host_tensors(w: Workload, pin: bool = False) -> Dict[str, object]:
    """The batch's inputs as CPU tensors (optionally page-locked for async copies)."""
    out = {}
    for f in INPUT_FIELDS:
        a = getattr(w, f)
        if a is None:
            out[f] = None
            continue
        t = _host_tensor(a, bf16=(f == "logits" and w.logits_dtype == BF16))
        out[f] = t.pin_memory() if pin else t
    return out


def device_tensors(w: Workload, device="cuda", host: Optional[Dict[str, object]] = None) -> Dict[str, object]:
    host = host or host_tensors(w)
    return {f: (None if t is None else t.to(device, non_blocking=True)) for f, t in host.items()}


@dataclasses.dataclass
class Outputs:
    out_tokens: object
    out_num_accepted: object
    counters: object
    status: object
    diag_accept_prob: Optional[object] = None
    diag_row_stats: Optional[object] = None
    workspace: Optional[object] = None
    telemetry: Optional[object] = None
    guarded: Optional[list] = None          # (whole allocation, elements in use) per guarded output

    def numpy(self) -> Dict[str, np.ndarray]:
        d = {"out_tokens": self.out_tokens, "out_num_accepted": self.out_num_accepted,
             "counters": self.counters, "status": self.status}
        if self.diag_accept_prob is not None:
            d["diag_accept_prob"] = self.diag_accept_prob
            d["diag_row_stats"] = self.diag_row_stats
        if self.telemetry is not None:
            d["telemetry"] = self.telemetry
        res = {}
        for k, t in d.items():
            t = t.cpu()
            if k in ("counters", "telemetry"):
                res[k] = t.view(dtype=__import__("torch").int64).numpy().view(np.uint64).copy()
            elif k == "status":
                res[k] = t.numpy().view(np.uint32).copy()
            else:
                res[k] = t.numpy().copy()
        if self.guarded is not None:
            res["guards_intact"] = self.guards_intact()
        return res

    def guards_intact(self) -> bool:
        """Whether the guard elements after every output still hold their fill pattern."""
        for base, n in self.guarded or []:
            tail = base.view(-1)[n:].cpu().numpy().view(np.uint8)
            if tail.size and not (tail == GUARD_BYTE).all():
                return False
        return True


GUARD_BYTE = 0xA5


def alloc_outputs(w: Workload, device="cuda", diag: bool = False, workspace: bool = True,
                  telemetry: Optional[bool] = None, guard: int = 0) -> Outputs:
    """Output tensors (and, with workspace=True, the verify's scratch: the request schedule).
    The per-position telemetry is allocated when asked for (default: with the diagnostics).
    guard > 0: every output is the front of a larger allocation whose last `guard` elements hold
    the byte 0xA5, so that Outputs.guards_intact() detects a write past an output's end."""
    import torch

    guarded = [] if guard > 0 else None

    def out(shape, fill, dtype):
        n = int(np.prod(shape))
        if not guard:
            return torch.full(shape, fill, dtype=dtype, device=device)
        base = torch.empty(n + guard, dtype=dtype, device=device)
        base.view(torch.uint8).fill_(GUARD_BYTE)
        t = base[:n].view(shape)
        t.fill_(fill)
        guarded.append((base, n))
        return t

    ws_bytes = _native.workspace_size(w.B, w.V) if workspace else 0
    return Outputs(
        out_tokens=out((w.T,), -7, torch.int32),
        out_num_accepted=out((w.B,), -7, torch.int32),
        counters=out((4,), 0, torch.int64),
        status=out((w.B,), 0, torch.int32),
        diag_accept_prob=out((max(w.N, 1),), float("nan"), torch.float32) if diag else None,
        diag_row_stats=out((max(w.T, 1), 2), float("nan"), torch.float32) if diag else None,
        workspace=torch.empty(ws_bytes, dtype=torch.uint8, device=device) if ws_bytes else None,
        telemetry=(out(_native.TELEMETRY_SHAPE, 0, torch.int64)
                   if (diag if telemetry is None else telemetry) else None),
        guarded=guarded,
    )


def verify(w: Workload, dev: Dict[str, object], out: Outputs, stream=None) -> None:
    """Queue one verify of batch `w` whose inputs are already in `dev`."""
    _native.specdec_verify(
        dev["logits"], dev["draft_ids"], dev["draft_probs"], dev["has_q"], dev["cu_num_draft"],
        w.B, w.V, w.max_k, dev["bitmask"], dev["temperature"], dev["uniforms"], dev["exp_noise"],
        out.out_tokens, out.out_num_accepted, out.counters, out.status,
        out.diag_accept_prob, out.diag_row_stats, workspace=out.workspace, stream=stream,
        telemetry=out.telemetry, top_k=dev.get("top_k"), top_p=dev.get("top_p"))


def run(w: Workload, device="cuda", diag: bool = True, workspace: bool = True, guard: int = 0,
        telemetry: Optional[bool] = None) -> Dict[str, np.ndarray]:
    """Copy, verify, synchronise, and return the outputs as numpy arrays (with guard > 0 also
    "guards_intact": whether every output's trailing guard elements are untouched)."""
    import torch

    dev = device_tensors(w, device)
    out = alloc_outputs(w, device, diag=diag, workspace=workspace, guard=guard, telemetry=telemetry)
    verify(w, dev, out)
    torch.cuda.synchronize()
    return out.numpy()
