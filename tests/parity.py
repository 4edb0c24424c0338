"""Element-by-element comparison of the CUDA path with the fp64 oracle.

Rules (written here, used by every parity test):

* Status bits, greedy tokens and greedy J: bit-exact.
* p_i(x_i): within P_TOL absolute of the oracle's fp64 value.
* Accept/reject decisions and drawn tokens: exact, except a FLAGGED disagreement:
  - chain rule: a decision may differ only at the first position where the two J differ,
    and only if the oracle's uniform lies within FLAG_TOL of that test's boundary p/q;
  - block rule: the accepted lengths may differ only if the survival test of the longer
    one lies within FLAG_TOL of its boundary (the test that one side passed and the
    other did not);
  - a drawn token may differ only if the GPU's token has positive weight and the
    uniform lies within FLAG_TOL of that token's interval [C_{k-1}/S, C_k/S] of the
    oracle's CDF -- the CDF of the distribution the GPU drew from: the residual, or p
    itself where the GPU (and not the oracle) found a zero residual by rounding; where
    only the oracle's residual is exactly zero, the GPU's token must have p > 0;
  - the zero-residual warning (decided by rounding) may differ: flagged.
  Anything else is a hard failure.  Flagged counts are reported per workload, together
  with the count the literal rule gives (every uniform within FLAG_TOL of any decision
  boundary or of any boundary of the oracle's CDF), and on every measured workload the
  flagged count must stay within MAX_FLAG_FRACTION of its rows (B * (gamma + 1) per
  round), with no floor: 1e-4 of 500 rows allows no flag at all.

The oracle runs in a spawn-started process pool over memory-mapped inputs for the large
workloads, so it never forks a process that holds a CUDA context.
"""
from __future__ import annotations

import multiprocessing as mp
import os
import tempfile

import numpy as np

P_TOL = 1e-6
FLAG_TOL = 1e-5
MAX_FLAG_FRACTION = 1e-4


def assert_flag_budget(flagged: int, rows: int, summary=None):
    """The stated bound on flagged rows: at most MAX_FLAG_FRACTION of them, no floor."""
    assert flagged <= MAX_FLAG_FRACTION * rows, (flagged, rows, summary)


_W = {}


def _init_worker(folder, mode="chain"):
    import sys
    here = os.path.dirname(os.path.abspath(__file__))
    root = os.path.dirname(here)
    for p in (root, here):
        if p not in sys.path:
            sys.path.insert(0, p)
    for name in ("logits", "q", "drafts", "T", "u", "gpu_tokens", "gpu_J", "gammas"):
        _W[name] = np.load(os.path.join(folder, name + ".npy"), mmap_mode="r")
    _W["mode"] = mode


def _oracle_one(b):
    from oracle import specdec_oracle as so
    logits = np.asarray(_W["logits"][b], dtype=np.float64)
    q = np.asarray(_W["q"][b], dtype=np.float64) if _W["q"].size else None
    drafts = np.asarray(_W["drafts"][b])
    T = float(_W["T"][b])
    u = np.asarray(_W["u"][b], dtype=np.float64)
    gamma = len(drafts)
    if _W["mode"] == "varlen":  # the extra token's uniform sits at slot gamma_b
        gb = int(_W["gammas"][b])
        r = so.verify_chain_varlen_sequence(logits, q, drafts, T, u, gb, want_cdf=True)
        gamma = gb
    else:
        verify = so.verify_block_sequence if _W["mode"] == "block" else so.verify_chain_sequence
        r = verify(logits, q, drafts, T, u, want_cdf=True)
    out = {
        "tokens": r["tokens"], "J": r["J"], "status": r["status"], "p_draft": r["p_draft"],
        "margins": r["margins"], "greedy": r["greedy"], "lit_draw": False,
        "y_interval": None, "y_weight": None, "yp_interval": None, "yp_weight": None,
    }
    if "cdf" in r:
        C, S = r["cdf"], r["S"]
        uu = u[gamma]
        t = uu * S
        k = int(np.searchsorted(C, t, side="right"))
        lo = C[k - 1] if k > 0 else 0.0
        hi = C[k] if k < len(C) else S
        out["lit_draw"] = bool(min(t - lo, hi - t) < FLAG_TOL * S)
        gJ = int(_W["gpu_J"][b])
        if gJ == r["J"]:
            gy = int(_W["gpu_tokens"][b][gJ])
            if 0 <= gy < len(C):
                a = C[gy - 1] if gy > 0 else 0.0
                out["y_interval"] = (a / S, C[gy] / S)
                out["y_weight"] = C[gy] - a
                Cp = r["pcdf"]
                ap = Cp[gy - 1] if gy > 0 else 0.0
                out["yp_interval"] = (ap / Cp[-1], Cp[gy] / Cp[-1])
                out["yp_weight"] = Cp[gy] - ap
    return out


def run_oracle_chain(logits, q, drafts, T, u, gpu_tokens, gpu_J, workers=None, mode="chain", gammas=None):
    """Oracle summaries for every sequence (numpy inputs; logits already widened to
    float32 for bf16 workloads, which is exact).  mode: "chain", "block" or "varlen"
    (gammas [B]: the drafts each sequence verifies)."""
    B = logits.shape[0]
    with tempfile.TemporaryDirectory() as folder:
        arrays = {"logits": logits, "q": q if q is not None else np.zeros(0, np.float32),
                  "drafts": drafts, "T": T, "u": u, "gpu_tokens": gpu_tokens, "gpu_J": gpu_J,
                  "gammas": gammas if gammas is not None else np.zeros(0, np.int32)}
        for k, v in arrays.items():
            np.save(os.path.join(folder, k + ".npy"), np.ascontiguousarray(v))
        nw = workers if workers is not None else min(os.cpu_count() or 1, 16)
        if nw <= 1 or B <= 4:
            _init_worker(folder, mode)
            res = [_oracle_one(b) for b in range(B)]
            _W.clear()
            return res
        ctx = mp.get_context("spawn")
        with ctx.Pool(nw, initializer=_init_worker, initargs=(folder, mode)) as pool:
            return pool.map(_oracle_one, range(B), chunksize=max(1, B // (4 * nw)))


class ParityReport:
    def __init__(self, name):
        self.name = name
        self.sequences = 0
        self.rows = 0
        self.draws = 0
        self.flag_decision = 0
        self.flag_draw = 0
        self.literal = 0
        self.accepted = 0
        self.failures = []
        self.max_p_err = 0.0
        self.flag_details = []  # per flagged draw: distance of u from the GPU token's interval

    @property
    def flagged(self):
        return self.flag_decision + self.flag_draw

    def summary(self) -> dict:
        return {
            "workload": self.name, "sequences": self.sequences, "rows": self.rows,
            "draws": self.draws, "flagged_decisions": self.flag_decision,
            "flagged_draws": self.flag_draw, "flagged_fraction_of_rows": self.flagged / max(self.rows, 1),
            "literal_rule_flags": self.literal, "max_abs_p_error": self.max_p_err,
            "mean_accepted": self.accepted / max(self.sequences, 1), "hard_failures": len(self.failures),
            "flagged_draw_details": self.flag_details[:20],
        }

    def fail(self, msg):
        if len(self.failures) < 20:
            self.failures.append(msg)
        else:
            self.failures.append("...")


def check_chain(report: ParityReport, gpu: dict, orc: list, u: np.ndarray, rule: str = "chain",
                extra_slot=None):
    """Compare one batch.  gpu: numpy tokens [B, g+1], num_accepted [B], status [B],
    p_draft [B, g] (optional).  rule: "chain" or "block" (which test decides a length);
    extra_slot [B]: the uniform slot of each sequence's extra token (default gamma)."""
    B, g1 = gpu["tokens"].shape
    gamma = g1 - 1
    for b in range(B):
        o = orc[b]
        report.sequences += 1
        report.rows += g1
        gt, gJ, gs = gpu["tokens"][b], int(gpu["num_accepted"][b]), int(gpu["status"][b])
        os_ = int(o["status"])
        if (gs & 0xFF) != (os_ & 0xFF) or (gs & 256) != (os_ & 256):
            report.fail(f"seq {b}: status gpu {gs} oracle {os_}")
            continue
        if os_ & 0xFF:
            if gJ != -1 or (gt != -1).any():
                report.fail(f"seq {b}: error sequence has outputs J={gJ} {gt}")
            continue
        if "p_draft" in gpu and not o["greedy"]:
            gp = gpu["p_draft"][b].astype(np.float64)
            op = o["p_draft"]
            ok = np.isfinite(op)
            if gJ == o["J"] and not np.array_equal(np.isnan(gp), np.isnan(op)):
                report.fail(f"seq {b}: p_draft evaluated positions differ {gp} vs {op}")
            if ok.any():
                err = float(np.max(np.abs(gp[ok] - op[ok])))
                report.max_p_err = max(report.max_p_err, err)
                if err > P_TOL:
                    report.fail(f"seq {b}: |p_draft error| {err:.3g} > {P_TOL}")
        if not o["greedy"]:
            tested = gamma if rule == "block" else min(o["J"] + 1, gamma)
            report.literal += int(np.sum(o["margins"][:tested] < FLAG_TOL)) + int(o["lit_draw"])
            report.draws += 1
        if o["greedy"]:
            if gJ != o["J"] or not np.array_equal(gt, o["tokens"]):
                report.fail(f"seq {b}: greedy mismatch gpu J={gJ} {gt} oracle J={o['J']} {o['tokens']}")
            report.accepted += o["J"]
            continue
        report.accepted += o["J"]
        if gJ != o["J"]:
            i = (max(gJ, o["J"]) - 1) if rule == "block" else min(gJ, o["J"])
            if 0 <= i < gamma and o["margins"][i] < FLAG_TOL:
                report.flag_decision += 1
            else:
                report.fail(f"seq {b}: J gpu {gJ} oracle {o['J']} margin {o['margins'][i] if 0 <= i < gamma else None}")
            continue
        J = gJ
        if not np.array_equal(gt[:J], o["tokens"][:J]) or (gt[J + 1:] != -1).any():
            report.fail(f"seq {b}: accepted prefix or padding differs {gt} vs {o['tokens']}")
            continue
        if gt[J] != o["tokens"][J]:
            uu = float(u[b, gamma if extra_slot is None else int(extra_slot[b])])
            gz, oz = bool(gs & 512), bool(os_ & 512)
            if gz and not oz:  # the GPU drew from p_J: its token's interval in p_J's CDF
                iv, w = o["yp_interval"], o["yp_weight"]
            elif oz and not gz:  # the exact residual is zero: any token of p_J > 0 is possible
                iv, w = (0.0, 1.0), o["yp_weight"]
            else:
                iv, w = o["y_interval"], o["y_weight"]
            if iv is not None and w is not None and w > 0 and iv[0] - FLAG_TOL <= uu <= iv[1] + FLAG_TOL:
                report.flag_draw += 1
                dist = 0.0 if iv[0] <= uu <= iv[1] else min(abs(uu - iv[0]), abs(uu - iv[1]))
                report.flag_details.append({"seq": b, "J": J, "u": uu, "outside_by": dist,
                                            "gpu": int(gt[J]), "oracle": int(o["tokens"][J]),
                                            "interval": [float(iv[0]), float(iv[1])]})
            else:
                report.fail(f"seq {b}: draw gpu {gt[J]} oracle {o['tokens'][J]} u {uu} gpu-interval {iv} "
                            f"zero-residual gpu {gz} oracle {oz}")
        elif (gs & 512) != (os_ & 512):
            report.flag_draw += 1  # the zero-residual warning alone, decided by rounding
