"""Chooses the Sinkhorn iteration count K with the oracle alone.

The KVarN page ("KVarN Nasil Calisir?", stage "Normalize Edilmis Onbellek")
says the row/column log-domain variance normalization is Sinkhorn-like but
gives no iteration count.  Rule used here: the smallest K whose decode-attention
error against exact fp16 attention (float64, no quantization) is within 1 %
(relative) of the error at K = 32, on a sample of the Llama-3-8B-like layer
workload (same distributions, fewer sequences).

Run:  python -m oracle.select_sinkhorn_iters   (prints one JSON line)
"""
from __future__ import annotations

import json
import sys
import time

import numpy as np

from oracle import kvref as R
from workloads import synth


def exact_attention(q, k, v, hq, hkv, scale):
    """float64 softmax attention over the fp16 cache, every token."""
    qd = q.astype(np.float64)
    kd = k.astype(np.float64)
    vd = v.astype(np.float64)
    B = q.shape[0]
    g = hq // hkv
    out = np.zeros((B, hq, 128))
    for b in range(B):
        for h in range(hq):
            s = kd[b, :, h // g, :] @ qd[b, h] * scale
            s = np.exp(s - s.max())
            out[b, h] = (s[:, None] * vd[b, :, h // g, :]).sum(0) / s.sum()
    return out


def main(argv=None):
    w = synth.scaled(synth.WORKLOADS["llama3_8b_layer"], batch=4, seq=4096)
    k, v = synth.kv(w)
    q = synth.queries(w)
    lens = synth.seq_lens(w).numpy()
    tables, num_pages = synth.block_tables(w)
    table = tables[0].numpy()
    k16, v16, q16 = k.numpy(), v.numpy(), q.numpy()
    scale = 1.0 / np.sqrt(128.0)
    ref = exact_attention(q16, k16, v16, w.hq, w.hkv, scale)
    errs = {}
    t0 = time.time()
    for iters in (0, 1, 2, 3, 4, 6, 8, 32):
        st = R.quantize_blocks(k16, v16, lens, table, num_pages, iters)
        o = R.decode_attention(q16, st["pool"], table, lens, st["tail_k"], st["tail_v"], w.hq,
                               w.hkv, scale, route=1)
        errs[iters] = float(np.linalg.norm(o - ref) / np.linalg.norm(ref))
    chosen = min(kk for kk in errs if kk > 0 and errs[kk] <= 1.01 * errs[32])
    print(json.dumps({"workload": synth.describe(w), "rel_err_by_iters": errs,
                      "chosen_iters": chosen, "seconds": round(time.time() - t0, 1)}))
    return 0


if __name__ == "__main__":
    sys.exit(main())
