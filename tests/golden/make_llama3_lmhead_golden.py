"""Writes tests/golden/llama3_lmhead_golden.npz: oracle values of the Llama-3-8B
lm_head workload (BT=4096, H=4096, V=128256, bf16, independent student and
teacher, 5% ignored rows, beta=0.5, T=1, batchmean), for the full-size GPU
parity test.

    python tests/golden/make_llama3_lmhead_golden.py

The inputs are drawn on the CPU by jsd_inputs (the workload's recipe); every
stored value comes from the float64 oracle alone (oracle.logits,
oracle.jsd_rows, oracle.row_weights), over every row of the batch:

* the batchmean loss and the per-row losses L_r (PR 1352 "Details": the loss
  is a per-row vector reduced afterwards);
* 64 rows of grad_weight = sum over all rows of dz^T X_s (PR 1429 "Summary":
  the product summed over every chunk), chosen at the first and last
  vocabulary ids, the last 256-column tile, 128-column boundaries and random
  ids;
* 8 rows of grad_input = dz W_s (one of them an ignored row, exactly 0);
* SHA-256 digests of the input tensors' bytes, so that the test can tell that
  it regenerated the same inputs.

The stored file comes from the machine that runs the GPU tests (an Arm host):
torch's CPU normal sampler does not give bit-identical draws across CPU
architectures, so a file written on another machine fails the digest check.
It takes about a minute on 16 cores and about 10 GB of host memory.
"""
from __future__ import annotations

import hashlib
import os
import sys
import time

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(os.path.dirname(HERE))
sys.path.insert(0, ROOT)
OUT = os.path.join(HERE, "llama3_lmhead_golden.npz")
BLOCK = 128


def digest(t) -> str:
    return hashlib.sha256(t.contiguous().view(-1).view(dtype=_u8()).numpy().tobytes()).hexdigest()


def _u8():
    import torch

    return torch.uint8


def selected_vocab(v: int, seed: int) -> np.ndarray:
    fixed = {0, 1, 127, 128, 255, 256, 4095, 4096, v // 2, v - 257, v - 256, v - 129, v - 128,
             v - 2, v - 1}
    fixed |= set(range(v - 256, v, 37))  # inside the last 256-column tile
    rng = np.random.default_rng(seed)
    while len(fixed) < 64:
        fixed.add(int(rng.integers(0, v)))
    return np.array(sorted(fixed), dtype=np.int64)


def main(out=OUT):
    import jsd_inputs
    import oracle

    w = jsd_inputs.WORKLOADS["llama3_lmhead"]
    t0 = time.time()
    x_s, w_s, x_t, w_t, labels = jsd_inputs.make_inputs(w, "cpu")
    digests = {k: digest(t) for k, t in
               (("x_s", x_s), ("w_s", w_s), ("x_t", x_t), ("w_t", w_t), ("labels", labels))}
    xs = x_s.double().numpy()
    ws = w_s.double().numpy()
    xt = x_t.double().numpy()
    wt = w_t.double().numpy()
    lab = labels.numpy()
    bt, v = w.bt, w.v
    wgt, valid, n = oracle.row_weights(lab, bt, v, w.reduction)
    J = selected_vocab(v, 4)
    rng = np.random.default_rng(5)
    ign = np.nonzero(~valid)[0]
    R = np.array(sorted({0, bt - 1, int(ign[0])} |
                        set(int(r) for r in rng.choice(bt, 5, replace=False))), dtype=np.int64)
    loss_rows = np.zeros(bt)
    gw_J = np.zeros((len(J), w.h_s))
    gi_R = np.zeros((len(R), w.h_s))
    for r0 in range(0, bt, BLOCK):
        r1 = min(bt, r0 + BLOCK)
        zs = oracle.logits(xs[r0:r1], ws)
        zt = oracle.logits(xt[r0:r1], wt)
        L, dA = oracle.jsd_rows(zs, zt, w.beta, w.temperature)
        vb = valid[r0:r1]
        loss_rows[r0:r1] = np.where(vb, L, 0.0)
        dz = dA * (wgt[r0:r1] / w.temperature)[:, None]
        dz[~vb] = 0.0
        gw_J += dz[:, J].T @ xs[r0:r1]
        for i, r in enumerate(R):
            if r0 <= r < r1:
                gi_R[i] = dz[r - r0] @ ws
        print(f"rows {r1}/{bt}  {time.time() - t0:.0f} s", flush=True)
    loss = float(loss_rows.sum() / n)
    np.savez_compressed(
        out, loss=np.float64(loss), loss_rows=loss_rows, vocab_ids=J,
        grad_weight_rows=gw_J.astype(np.float32), row_ids=R,
        grad_input_rows=gi_R.astype(np.float32), n_valid=np.int64(n),
        **{f"sha256_{k}": np.array(d) for k, d in digests.items()})
    print(f"wrote {out}: loss {loss:.9g}, n = {n}, {time.time() - t0:.0f} s")


if __name__ == "__main__":
    main(sys.argv[1] if len(sys.argv) > 1 else OUT)
