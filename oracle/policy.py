"""Per-block precision / caching policy (oracle; test infrastructure only).

Rules, from "6Bit-Diffusion" (technical summary sections 2.A-2.C; popular
summary sections 1-3):

* DMPQ: a block that was stable at t-1 (small Gamma_{t-1}) runs NVFP4, a
  volatile one runs INT8.
* TDC: if Delta_{t-1} and Delta_{t-2} are similar enough, skip the block and
  reuse the cached delta; an error accumulator forces a refresh once the
  accumulated predicted error exceeds a cap.
* PDR: before a delta is cached, an input whose max/mean outlier ratio is
  too high is recomputed in full precision (BF16) instead.
* After a skip, Gamma_{t-1} is missing, so the block restarts in INT8.

Readings where the pages are silent (listed with the code that takes them):
  (i)   a skip adds its predicted error 1 - cos to the accumulator;
  (ii)  cos >= cos_thr may skip; acc + (1 - cos) > err_cap forces a refresh;
        ratio > pdr_ratio forces BF16; Gamma >= gamma_thr picks INT8;
  (iii) a refresh is a normal compute under the rules below (INT8 after a
        skip, BF16 if PDR fires); refresh_bf16=True instead makes every
        refresh BF16 (the popular summary's "full precision" refresh);
  (iv)  the PDR test runs before computing, on the block input;
  (v)   one decision per block covers all its linear layers;
  (vi)  the first two computed steps never skip (no cosine yet);
  (vii) a statistic that is not a number (a corrupted or overflowed sum)
        fails its threshold test toward the safer path: a NaN cosine never
        skips, a NaN Gamma picks INT8 and a NaN input ratio picks BF16.

Decision of step s, then the fold of its statistics (if it computed):

    if n_computed >= 2 and cos >= cos_thr:
        if acc + (1 - cos) <= err_cap: SKIP; acc += 1 - cos; skipped_last = True
        else: REFRESH (a compute, flagged)
    compute: BF16 if ratio > pdr_ratio or NaN (or refresh and refresh_bf16)
             else INT8 if skipped_last or no Gamma yet
             else NVFP4 if Gamma < gamma_thr else INT8 (so a NaN Gamma: INT8)
    after a compute: Gamma <- new Gamma; cos <- cos(Delta_new, Delta_prev) if a
        previous delta existed; n_computed += 1; acc = 0; skipped_last = False
"""
from __future__ import annotations

from dataclasses import dataclass, field

SKIP, NVFP4, INT8, BF16 = "SKIP", "NVFP4", "INT8", "BF16"


@dataclass
class PolicyConfig:
    gamma_thr: float = 0.1
    cos_thr: float = 0.99
    err_cap: float = 0.05
    pdr_ratio: float = 30.0
    refresh_bf16: bool = False
    near_rel: float = 1e-6


@dataclass
class Decision:
    mode: str
    refresh: bool = False
    pdr: bool = False
    post_skip: bool = False
    near: bool = False          # a deciding statistic was within near_rel of its threshold


@dataclass
class PolicyState:
    n_computed: int = 0
    skipped_last: bool = False
    have_gamma: bool = False
    gamma: float = 0.0
    cos: float = 0.0
    acc: float = 0.0
    history: list = field(default_factory=list)


def _near(v: float, thr: float, rel: float) -> bool:
    return abs(v - thr) <= rel * abs(thr)


def decide(st: PolicyState, ratio: float, cfg: PolicyConfig) -> Decision:
    """Decision for the current step; updates the skip-side state (acc, skipped_last)."""
    near = False
    refresh = False
    if st.n_computed >= 2:
        near |= _near(st.cos, cfg.cos_thr, cfg.near_rel)
        if st.cos >= cfg.cos_thr:
            pred = st.acc + (1.0 - st.cos)
            near |= _near(pred, cfg.err_cap, cfg.near_rel)
            if pred <= cfg.err_cap:
                st.acc = pred
                st.skipped_last = True
                d = Decision(SKIP, near=near)
                st.history.append(d)
                return d
            refresh = True
    near |= _near(ratio, cfg.pdr_ratio, cfg.near_rel)
    pdr = not (ratio <= cfg.pdr_ratio)   # above the threshold, or not a number
    if pdr or (refresh and cfg.refresh_bf16):
        d = Decision(BF16, refresh=refresh, pdr=pdr, near=near)
    elif st.skipped_last or not st.have_gamma:
        d = Decision(INT8, refresh=refresh, post_skip=st.skipped_last, near=near)
    else:
        near |= _near(st.gamma, cfg.gamma_thr, cfg.near_rel)
        d = Decision(NVFP4 if st.gamma < cfg.gamma_thr else INT8, refresh=refresh, near=near)   # NaN: INT8
    st.history.append(d)
    return d


def fold(st: PolicyState, gamma: float, cos) -> None:
    """Fold the statistics of a computed step into the state."""
    st.gamma = gamma
    st.have_gamma = True
    if cos is not None and st.n_computed >= 1:
        st.cos = cos
    st.n_computed += 1
    st.acc = 0.0
    st.skipped_last = False


def run_trace(steps, cfg: PolicyConfig | None = None):
    """Run the policy over hand-made steps.

    ``steps`` is a list of dicts with key 'ratio' and, for computed steps,
    the statistics the compute produced: 'gamma' and optionally 'cos'.
    Returns the list of Decisions.
    """
    cfg = cfg or PolicyConfig()
    st = PolicyState()
    out = []
    for s in steps:
        d = decide(st, s["ratio"], cfg)
        out.append(d)
        if d.mode != SKIP:
            fold(st, s["gamma"], s.get("cos"))
    return out
