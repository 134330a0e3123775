"""Seeded synthetic inputs for the fused-linear JSD loss.

This module only draws random tensors of the right shapes, dtypes and
structure; it holds none of the loss arithmetic. The same tensors are fed to
the CUDA library and to the CPU oracle.

Recipe (every workload): a torch generator seeded with the workload's seed
draws, in this order, X_s [BT x H_s] ~ N(0, 1), W_s [V x H_s] ~ N(0, 1/H_s),
X_t [BT x H_t] ~ N(0, 1) and W_t [V x H_t] ~ N(0, 1/H_t) in float32; each is
then cast to the workload dtype. Labels come from a separate CPU generator with
the same seed: uniform in [0, V), then the first floor(frac*BT) rows of a
random permutation are set to ignore_index (-100).

The hidden states and lm_head weights of a real model are not needed: the
pages measure on synthetic shapes only (H=4096, V=128256, bf16).
"""
from __future__ import annotations

import dataclasses
import math

import torch

IGNORE_INDEX = -100


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    seed: int
    bt: int
    h_s: int
    h_t: int
    v: int
    dtype: str  # "fp32" | "bf16"
    beta: float = 0.5
    temperature: float = 1.0
    reduction: str = "batchmean"
    ignore_frac: float = 0.0
    tie: str = "none"  # "none" | "self" (X_t=X_s, W_t=W_s) | "padded"
    pad_frac: float = 0.0  # fraction of trailing vocab rows zeroed in W_s and W_t
    spike: int = 0  # > 0: the first `spike` tokens get a shared logit offset (below)

    @property
    def torch_dtype(self):
        return torch.float32 if self.dtype == "fp32" else torch.bfloat16

    def flops(self) -> float:
        """Dense FLOPs of one forward+backward: 2*BT*V*(3*H_s + H_t)."""
        return 2.0 * self.bt * self.v * (3 * self.h_s + self.h_t)


WORKLOADS = {
    # tiny fp32 case the oracle finishes instantly
    "tiny_fp32": Workload("tiny_fp32", 1, 64, 128, 128, 1000, "fp32"),
    # self-distillation: every element ties
    "ties_self": Workload("ties_self", 2, 1024, 4096, 4096, 32000, "bf16", tie="self"),
    # independent teacher weights; the last 10% of vocab rows are zero in both
    "ties_padded": Workload("ties_padded", 2, 1024, 4096, 4096, 32000, "bf16",
                            tie="padded", pad_frac=0.1),
    # multi-block vocabulary with a partial trailing block, 10% ignored rows
    "multiblock": Workload("multiblock", 3, 2048, 2048, 2048, 40960, "bf16", ignore_frac=0.1),
    # Llama-3-8B lm_head shape, 5% ignored rows
    "llama3_lmhead": Workload("llama3_lmhead", 4, 4096, 4096, 4096, 128256, "bf16",
                              ignore_frac=0.05),
    # student H=4096, teacher H=8192
    "large_teacher": Workload("large_teacher", 5, 8192, 4096, 8192, 128256, "bf16",
                              beta=0.1, temperature=2.0, ignore_frac=0.05),
    # the pages' benchmark shape: BT=8192, H=4096, V=128256, bf16
    "headline": Workload("headline", 6, 8192, 4096, 4096, 128256, "bf16"),
    # the headline's H and V with BT=1024 (small enough for full profiler captures)
    "headline_bt1024": Workload("headline_bt1024", 7, 1024, 4096, 4096, 128256, "bf16"),
    # the headline's BT and H with a quarter of V (about 2 GB on the device):
    # every kernel of a step keeps the headline's schedule, and its work and
    # traffic per launch scale with V, so profiler counters taken here scale
    # to the headline by 4
    "headline_v32k": Workload("headline_v32k", 8, 8192, 4096, 4096, 32064, "bf16"),
    # the headline's V with a small H and BT (about 1.5 GB on the device): the
    # row kernel, which does not depend on H, at full row length
    "rows_v128k": Workload("rows_v128k", 9, 2048, 512, 512, 128256, "bf16"),
}


def _randn(shape, std, gen, device):
    t = torch.empty(shape, dtype=torch.float32, device=device)
    t.normal_(0.0, std, generator=gen)
    return t


def make_labels(bt: int, v: int, ignore_frac: float, seed: int) -> torch.Tensor | None:
    """int64 labels [BT]: uniform in [0, V); floor(frac*BT) rows set to -100."""
    if ignore_frac <= 0.0:
        return None
    g = torch.Generator().manual_seed(seed)
    labels = torch.randint(0, v, (bt,), generator=g, dtype=torch.int64)
    n_ign = int(math.floor(ignore_frac * bt))
    perm = torch.randperm(bt, generator=g)
    labels[perm[:n_ign]] = IGNORE_INDEX
    return labels


def make_inputs(w: Workload, device: str = "cpu"):
    """Draw (x_s, w_s, x_t, w_t, labels) for a workload on ``device``.

    The float tensors are created on ``device`` (a CUDA generator is used for a
    CUDA device, so the numbers differ from a CPU draw with the same seed, but
    each draw is reproducible). Labels are always drawn on the CPU and moved.
    """
    gen = torch.Generator(device=device).manual_seed(w.seed)
    x_s = _randn((w.bt, w.h_s), 1.0, gen, device)
    w_s = _randn((w.v, w.h_s), 1.0 / math.sqrt(w.h_s), gen, device)
    if w.tie == "self":
        x_t, w_t = x_s, w_s
    else:
        x_t = x_s if w.tie == "padded" else _randn((w.bt, w.h_t), 1.0, gen, device)
        w_t = _randn((w.v, w.h_t), 1.0 / math.sqrt(w.h_t), gen, device)
    if w.pad_frac > 0.0:
        first = w.v - int(round(w.pad_frac * w.v))
        w_s[first:] = 0.0
        w_t[first:] = 0.0
    if w.spike > 0:
        # Hidden column 0 is 1 in both models and the first `spike` vocab rows
        # carry a weight of 8 there and 1% of the random weights elsewhere
        # (the teacher's with an independent 1% perturbation), so these tokens
        # lead both distributions by about 4 logit units or more and stay close to
        # each other, while every other token keeps an N(0, 1) logit that
        # differs between the models.
        k = w.spike
        x_s[:, 0] = 1.0
        w_s[:k] *= 0.01
        w_s[:k, 0] = 8.0
        if w.tie != "self":
            if x_t is not x_s:
                x_t[:, 0] = 1.0
            w_t[:k] = w_s[:k] + 0.01 * _randn((k, w.h_t), 1.0 / math.sqrt(w.h_t), gen, device)
            w_t[:k, 0] = 8.0
    dt = w.torch_dtype
    x_s, w_s = x_s.to(dt), w_s.to(dt)
    if w.tie == "self":
        x_t, w_t = x_s, w_s
    else:
        x_t = x_s if w.tie == "padded" else x_t.to(dt)
        w_t = w_t.to(dt)
    labels = make_labels(w.bt, w.v, w.ignore_frac, w.seed)
    if labels is not None:
        labels = labels.to(device)
    return x_s, w_s, x_t, w_t, labels


def custom(name: str, seed: int, bt: int, h_s: int, v: int, dtype: str = "bf16",
           h_t: int | None = None, **kw) -> Workload:
    """A workload of arbitrary shape with the same recipe (for small and odd shapes)."""
    return Workload(name, seed, bt, h_s, h_s if h_t is None else h_t, v, dtype, **kw)


def make_partial_ties(bt: int, h: int, v: int, dtype: str, seed: int, *, temperature: float,
                      diff_cols, n_full: int, n_free: int, ignore_frac: float = 0.0,
                      device: str = "cpu"):
    """Inputs whose rows tie (student and teacher log-probabilities exactly
    equal) at most columns but not all.

    Ties that hold exactly in any arithmetic need bitwise-equal log-normalisers
    on both sides, so the logits of the two models agree everywhere except in
    a few columns ``diff_cols`` whose logits lie so far below the row maximum
    (about 45 scaled units) that they cannot change a float64 or float32 sum of
    exponentials, yet still give normal float32 probabilities:

    * X_s ~ N(0, 1) [BT x H] and W_s ~ N(0, 1/H) [V x H] in float32, drawn in
      that order from a generator seeded with ``seed``; hidden column 0 of W_s
      is then set to 0.
    * Vocabulary rows ``diff_cols`` of W_s are 0 except hidden column 0, which
      is c_s; in W_t = W_s it is c_t. With X[:, 0] = 8 their logits are exactly
      8 c_s and 8 c_t (representable in bf16): c_s, c_t = -5, -4.5 at T = 1
      and -12, -11 at T = 2 (scaled logits -40 / -36 and -48 / -44).
    * Row kinds (a seeded permutation scatters them): "partial" rows have
      X_t = X_s and X[:, 0] = 8, so they tie everywhere except ``diff_cols``;
      ``n_full`` "full" rows have X[:, 0] = 0, so every logit of both models
      is equal and the row ties everywhere; ``n_free`` "free" rows get an
      independent teacher row X_t ~ N(0, 1) (X_t[:, 0] = 8), so they tie
      nowhere and carry ordinary loss and gradient.
    * Labels as in make_labels (``ignore_frac`` of the rows ignored).

    Returns ((x_s, w_s, x_t, w_t, labels), kinds) with kinds an array of
    "partial" / "full" / "free" per row.
    """
    import numpy as np

    if temperature == 1.0:
        c_s, c_t = -5.0, -4.5
    elif temperature == 2.0:
        c_s, c_t = -12.0, -11.0
    else:
        raise ValueError("the construction is calibrated for T = 1 and T = 2")
    gen = torch.Generator(device=device).manual_seed(seed)
    x_s = _randn((bt, h), 1.0, gen, device)
    w_s = _randn((v, h), 1.0 / math.sqrt(h), gen, device)
    x_free = _randn((bt, h), 1.0, gen, device)
    perm = torch.randperm(bt, generator=torch.Generator().manual_seed(seed + 1))
    kinds = np.array(["partial"] * bt, dtype=object)
    full = perm[:n_full]
    free = perm[n_full:n_full + n_free]
    kinds[full.numpy()] = "full"
    kinds[free.numpy()] = "free"
    cols = torch.as_tensor(list(diff_cols), dtype=torch.int64)
    w_s[:, 0] = 0.0
    w_s[cols] = 0.0
    w_t = w_s.clone()
    w_s[cols, 0] = c_s
    w_t[cols, 0] = c_t
    x_s[:, 0] = 8.0
    x_s[full.to(device), 0] = 0.0
    x_t = x_s.clone()
    x_t[free.to(device)] = x_free[free.to(device)]
    x_t[free.to(device), 0] = 8.0
    dt = torch.float32 if dtype == "fp32" else torch.bfloat16
    labels = make_labels(bt, v, ignore_frac, seed)
    if labels is not None:
        labels = labels.to(device)
    return (x_s.to(dt), w_s.to(dt), x_t.to(dt), w_t.to(dt), labels), kinds


def make_distributions(rows: int, v: int, dtype: str, seed: int, *, logspace: bool,
                       scale: float = 2.0, tied_rows: int = 0, tied_frac: float = 0.0,
                       ignore_frac: float = 0.0, device: str = "cpu"):
    """Two [rows x V] distributions for the distance paths: softmax (or
    log_softmax when ``logspace``) of seeded N(0, scale^2) scores, computed in
    float32 and cast to the dtype. The first ``tied_rows`` rows of the second
    tensor equal the first's; in the other rows the trailing ``tied_frac`` of
    the vocabulary is copied from the first tensor (padded-vocabulary style
    ties). Returns (a, b, labels)."""
    g = torch.Generator(device=device).manual_seed(seed)
    sa = _randn((rows, v), scale, g, device)
    sb = _randn((rows, v), scale, g, device)
    f = torch.log_softmax if logspace else torch.softmax
    a = f(sa, dim=-1).to(torch.float32 if dtype == "fp32" else torch.bfloat16)
    b = f(sb, dim=-1).to(a.dtype)
    if tied_rows:
        b[:tied_rows] = a[:tied_rows]
    if tied_frac > 0.0:
        k = v - int(round(tied_frac * v))
        b[tied_rows:, k:] = a[tied_rows:, k:]
    labels = make_labels(rows, v, ignore_frac, seed)
    if labels is not None:
        labels = labels.to(device)
    return a.contiguous(), b.contiguous(), labels


def make_ce_inputs(bt: int, h: int, v: int, dtype: str, seed: int, *, ignore_frac: float = 0.0,
                   device: str = "cpu"):
    """Hidden states x [BT x H] ~ N(0, 1), lm_head weight w [V x H] ~ N(0, 1/H)
    (float32, cast to the dtype) and int64 labels uniform in [0, V) with
    floor(frac*BT) rows set to -100: the cross-entropy path's inputs."""
    g = torch.Generator(device=device).manual_seed(seed)
    x = _randn((bt, h), 1.0, g, device)
    w = _randn((v, h), 1.0 / math.sqrt(h), g, device)
    dt = torch.float32 if dtype == "fp32" else torch.bfloat16
    lg = torch.Generator().manual_seed(seed)
    labels = torch.randint(0, v, (bt,), generator=lg, dtype=torch.int64)
    n_ign = int(math.floor(ignore_frac * bt))
    if n_ign:
        labels[torch.randperm(bt, generator=lg)[:n_ign]] = IGNORE_INDEX
    return x.to(dt), w.to(dt), labels.to(device)
