"""The synthetic verification workloads.

Shapes, dtypes, logit distributions and temperatures of the five workloads the
library is measured on. The pages ("Accelerating Large Language Model Decoding
with Speculative Sampling", §6.1) evaluate on XSum and HumanEval with Chinchilla;
neither the datasets nor the weights exist here, so seeded Gaussian logits with
a controlled draft/target gap stand in for them.
"""

from __future__ import annotations

from dataclasses import dataclass, replace


@dataclass(frozen=True)
class Workload:
    name: str
    B: int                  # sequences verified per step
    K: int                  # draft tokens per sequence (lookahead)
    V: int                  # vocabulary size
    dtype: str              # "bf16" or "f32" logits
    target_std: float       # target logits ~ N(0, target_std^2)
    draft_noise_std: float  # draft logits = target + N(0, draft_noise_std^2)
    temperature: float      # decoding temperature applied to both p and q
    peaks: int = 0          # per target row, this many random ids get +peak_boost
    peak_boost: float = 0.0
    seed: int = 0
    steps: int = 1          # verify steps the workload is defined over

    @property
    def elem_bytes(self) -> int:
        return 2 if self.dtype == "bf16" else 4

    def ideal_bytes_per_step(self) -> int:
        """(2K+1) rows streamed once plus two rows re-read for sampling, per sequence."""
        return self.B * (2 * self.K + 3) * self.V * self.elem_bytes

    def draft_positions(self) -> int:
        return self.B * self.K

    def describe(self) -> str:
        peak = f", {self.peaks} peaks +{self.peak_boost:g}" if self.peaks else ""
        return (f"B={self.B},K={self.K},V={self.V},{self.dtype},target N(0,{self.target_std:g}^2)"
                f",draft noise {self.draft_noise_std:g},T={self.temperature:g}{peak}")


WORKLOADS = {
    "c1": Workload("b1-k4-v1000-f32", B=1, K=4, V=1000, dtype="f32", target_std=2.0,
                   draft_noise_std=0.5, temperature=1.0, seed=1000, steps=1),
    "c2": Workload("b8-k4-v32000-bf16", B=8, K=4, V=32000, dtype="bf16", target_std=3.0,
                   draft_noise_std=1.0, temperature=1.0, seed=1001, steps=1000),
    "c3": Workload("b64-k8-v128256-bf16-peaks", B=64, K=8, V=128256, dtype="bf16",
                   target_std=3.0, draft_noise_std=0.7, temperature=0.8, peaks=32,
                   peak_boost=8.0, seed=1002, steps=200),
    "c4": Workload("b256-k4-v256000-f32", B=256, K=4, V=256000, dtype="f32",
                   target_std=2.5, draft_noise_std=1.5, temperature=1.0, seed=1003,
                   steps=20),
}

SWEEP_K = (1, 2, 4, 8, 16)
SWEEP_NOISE = (0.1, 0.5, 1.0, 2.0)


def sweep_workload(k: int, noise: float) -> Workload:
    ki = SWEEP_K.index(k)
    ni = SWEEP_NOISE.index(noise)
    return Workload(f"sweep-b32-k{k}-v151936-bf16-noise{noise:g}", B=32, K=k, V=151936,
                    dtype="bf16", target_std=3.0, draft_noise_std=noise, temperature=1.0,
                    seed=2000 + 10 * ki + ni, steps=1)


def get_workload(name: str) -> Workload:
    """`c1`..`c4`, or `sweep-k{K}-n{noise}` for one acceptance-sweep cell."""
    if name in WORKLOADS:
        return WORKLOADS[name]
    if name.startswith("sweep-k"):
        k_str, n_str = name[len("sweep-k"):].split("-n")
        return sweep_workload(int(k_str), float(n_str))
    raise KeyError(name)


def shrink(w: Workload, **kw) -> Workload:
    """A copy with some fields replaced (used for small parity cases of a workload)."""
    return replace(w, **kw)


@dataclass(frozen=True)
class LMHeadWorkload:
    """Inputs of the scoring step's final projection: N hidden states of width
    D against a V-token projection, logits of standard deviation `logit_std`."""
    name: str
    N: int
    D: int
    V: int
    temperature: float
    logit_std: float
    seed: int

    def flops(self) -> int:
        return 2 * self.N * self.D * self.V

    def weight_bytes(self) -> int:
        return self.V * self.D * 2


# The target call of the 64x8x128256 workload: 64 sequences x 9 scored
# prefixes, a model width of 8192 and the workload's vocabulary and temperature.
LMHEAD_WORKLOADS = {
    "lmhead-c3": LMHeadWorkload("lmhead-n576-d8192-v128256-bf16", N=576, D=8192, V=128256,
                                temperature=0.8, logit_std=3.0, seed=3003),
}
