"""Element-by-element comparison of the GPU library's outputs with the CPU oracle's
(TEST INFRASTRUCTURE ONLY).

Rules (the tolerance the verify step is held to):
  * tokens, accepted lengths and counters are bit-exact, except from the first position
    of a request where the decision is within floating-point reach of a tie:
      - an acceptance test with |u - alpha_oracle| < 1e-6, or
      - a sampled token (recovered / bonus) whose race top-two scores differ by less than
        1e-6 relative;
    such a request is excluded from that position onward and its contribution to A is
    left out of the A check;
  * R, I, D are always exact; statuses are exact;
  * alpha of every draft both sides tested and the row statistics (m, S) agree within
    1e-5 relative.
"""
from __future__ import annotations

import dataclasses
from typing import List

import numpy as np

U_BAND = 1e-6
MARGIN_BAND = 1e-6
TOPP_BAND = 1e-6      # top-p: |mass above the boundary - top_p| (the kernel sums in fixed point)
P_RTOL = 1e-5


@dataclasses.dataclass
class ParityReport:
    requests: int = 0
    excluded_requests: int = 0
    excluded_positions: int = 0
    token_mismatches: List[tuple] = dataclasses.field(default_factory=list)
    accepted_mismatches: List[tuple] = dataclasses.field(default_factory=list)
    status_mismatches: List[tuple] = dataclasses.field(default_factory=list)
    counter_mismatch: str = ""
    alpha_max_rel: float = 0.0
    alpha_bad: List[tuple] = dataclasses.field(default_factory=list)
    row_m_max_rel: float = 0.0
    row_S_max_rel: float = 0.0
    row_bad: List[tuple] = dataclasses.field(default_factory=list)
    telemetry_mismatch: str = ""
    compared_tokens: int = 0

    @property
    def ok(self) -> bool:
        return not (self.token_mismatches or self.accepted_mismatches or self.status_mismatches
                    or self.counter_mismatch or self.alpha_bad or self.row_bad or self.telemetry_mismatch)

    def summary(self) -> str:
        return (f"requests={self.requests} excluded_requests={self.excluded_requests} "
                f"excluded_positions={self.excluded_positions} compared_tokens={self.compared_tokens} "
                f"token_mismatches={len(self.token_mismatches)} accepted_mismatches={len(self.accepted_mismatches)} "
                f"status_mismatches={len(self.status_mismatches)} counters='{self.counter_mismatch}' "
                f"alpha_max_rel={self.alpha_max_rel:.3g} row_m_max_rel={self.row_m_max_rel:.3g} "
                f"row_S_max_rel={self.row_S_max_rel:.3g} alpha_bad={len(self.alpha_bad)} row_bad={len(self.row_bad)} "
                f"telemetry='{self.telemetry_mismatch}'")


def _rel(a, b):
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    return np.abs(a - b) / np.maximum(np.abs(b), 1e-30)


def compare(w, gpu: dict, ref: dict, counters_before=(0, 0, 0, 0)) -> ParityReport:
    """w: the host Workload; gpu: numpy outputs of the library (device.run); ref: oracle result."""
    rep = ParityReport(requests=w.B)
    cu = w.cu_num_draft
    greedy = ~(w.temperature > 0) | ~np.isfinite(w.temperature) | (
        (w.temperature > 0) & (w.temperature < np.float32(1.17549435e-38)))
    excluded_A_gpu = 0
    excluded_A_ref = 0
    excluded_pairs = []          # (oracle a_b, library a_b) of requests cut at a near-tie
    g_tok, r_tok = gpu["out_tokens"], ref["out_tokens"]
    g_acc, r_acc = gpu["out_num_accepted"], ref["out_num_accepted"]
    for b in range(w.B):
        k = int(cu[b + 1] - cu[b]) if cu[b + 1] >= cu[b] else -1
        if int(gpu["status"][b]) != int(ref["status"][b]):
            rep.status_mismatches.append((b, int(gpu["status"][b]), int(ref["status"][b])))
        if k < 0:
            continue
        row0 = int(cu[b]) + b
        a_ref = int(r_acc[b])
        # first position that sits within floating-point reach of a tie (oracle's view)
        cut = None
        if not greedy[b] and not (int(ref["status"][b]) & (8 | 16)):
            for j in range(min(a_ref, k - 1) + 1 if k > 0 else 0):
                al = ref["alpha"][int(cu[b]) + j]
                if np.isfinite(al) and abs(float(w.uniforms[row0 + j]) - al) < U_BAND:
                    cut = j
                    break
            if cut is None:
                t1, t2 = ref["emit_top1"][b], ref["emit_top2"][b]
                if np.isfinite(t1) and t1 > 0 and (t1 - t2) / t1 < MARGIN_BAND:
                    cut = a_ref
        # a row whose top-p boundary sits within floating-point reach of top_p (oracle's view)
        tpm = ref.get("top_p_margin")
        if tpm is not None and not greedy[b] and not (int(ref["status"][b]) & (8 | 16)):
            for j in range(min(a_ref, k) + 1):
                if np.isfinite(tpm[row0 + j]) and tpm[row0 + j] < TOPP_BAND and (cut is None or j < cut):
                    cut = j
                    break
        if cut is not None:
            rep.excluded_requests += 1
            rep.excluded_positions += k + 1 - cut
            excluded_A_gpu += int(g_acc[b])
            excluded_A_ref += a_ref
            excluded_pairs.append((a_ref, int(g_acc[b])))
            for j in range(cut):
                rep.compared_tokens += 1
                if g_tok[row0 + j] != r_tok[row0 + j]:
                    rep.token_mismatches.append((b, j, int(g_tok[row0 + j]), int(r_tok[row0 + j])))
            continue
        if int(g_acc[b]) != a_ref:
            rep.accepted_mismatches.append((b, int(g_acc[b]), a_ref))
        for j in range(k + 1):
            rep.compared_tokens += 1
            if g_tok[row0 + j] != r_tok[row0 + j]:
                rep.token_mismatches.append((b, j, int(g_tok[row0 + j]), int(r_tok[row0 + j])))

    gc = np.asarray(gpu["counters"], dtype=np.int64) - np.asarray(counters_before, dtype=np.int64)
    rc = np.asarray(ref["counters"], dtype=np.int64)
    if list(gc[:3]) != list(rc[:3]):
        rep.counter_mismatch = f"R/I/D gpu={list(gc[:3])} oracle={list(rc[:3])}"
    elif int(gc[3]) - excluded_A_gpu != int(rc[3]) - excluded_A_ref:
        rep.counter_mismatch = f"A (outside exclusions) gpu={int(gc[3]) - excluded_A_gpu} oracle={int(rc[3]) - excluded_A_ref}"

    if gpu.get("telemetry") is not None and ref.get("telemetry") is not None:
        # drafts and eligible drafts by position are exact; accepted-through counts and the
        # histogram are exact outside the excluded requests, whose library a_b replaces the oracle's
        gt = np.asarray(gpu["telemetry"], dtype=np.int64).reshape(4, -1)
        want = np.asarray(ref["telemetry"], dtype=np.int64).reshape(4, -1).copy()
        for a_r, a_g in excluded_pairs:
            want[2, :a_r] -= 1
            want[3, a_r] -= 1
            want[2, :a_g] += 1
            want[3, a_g] += 1
        if gt.shape != want.shape or not np.array_equal(gt, want):
            bad = [(int(r), int(j), int(gt[r, j]), int(want[r, j])) for r, j in zip(*np.nonzero(gt != want))][:8]
            rep.telemetry_mismatch = f"(row, position, library, oracle): {bad}"

    if "diag_accept_prob" in gpu:
        ga = gpu["diag_accept_prob"][: w.N].astype(np.float64)
        ra = ref["alpha"]
        both = np.isfinite(ga) & np.isfinite(ra)
        if both.any():
            err = np.abs(ga[both] - ra[both]) / np.maximum(np.abs(ra[both]), 1e-30)
            # alpha within 1e-5 relative, or within fp32 resolution of tiny values
            bad = (err > P_RTOL) & (np.abs(ga[both] - ra[both]) > 1e-12)
            rep.alpha_max_rel = float(np.max(np.where(np.abs(ga[both] - ra[both]) > 1e-12, err, 0.0)))
            if bad.any():
                idx = np.flatnonzero(both)[bad]
                rep.alpha_bad = [(int(i), float(ga[i]), float(ra[i])) for i in idx[:20]]
        gr = gpu["diag_row_stats"][: w.T].astype(np.float64)
        rm, rS = ref["row_m"], ref["row_S"]
        bm = np.isfinite(gr[:, 0]) & np.isfinite(rm)
        if bm.any():
            em = np.abs(gr[bm, 0] - rm[bm]) / np.maximum(np.abs(rm[bm]), 1.0)
            rep.row_m_max_rel = float(em.max())
            badm = em > P_RTOL
            if badm.any():
                idx = np.flatnonzero(bm)[badm]
                rep.row_bad += [("m", int(i), float(gr[i, 0]), float(rm[i])) for i in idx[:20]]
        bS = np.isfinite(gr[:, 1]) & np.isfinite(rS)
        if bS.any():
            eS = _rel(gr[bS, 1], rS[bS])
            rep.row_S_max_rel = float(eS.max())
            badS = eS > P_RTOL
            if badS.any():
                idx = np.flatnonzero(bS)[badS]
                rep.row_bad += [("S", int(i), float(gr[i, 1]), float(rS[i])) for i in idx[:20]]
        # rows read by one side only
        read_g = np.isfinite(gr[:, 0]) | (gr[:, 0] == -np.inf)
        read_r = np.isfinite(rm) | (rm == -np.inf)
        if not np.array_equal(read_g, read_r):
            diff = np.flatnonzero(read_g != read_r)
            rep.row_bad += [("read", int(i), bool(read_g[i]), bool(read_r[i])) for i in diff[:20]]
    return rep
