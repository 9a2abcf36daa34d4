"""Print the ablation table (markdown): per variant and workload generator, stored bytes per
token-head, reconstruction error of the non-final loops and of the reference, and the error
of the attention output against attention over the unquantised states.

    python tests/ablation_table.py [n_tokens]

fp64, on the CPU, from the oracle's steps (tests/ablation.py); seeded synthetic states of
sequence 0, kv-heads 0-1, K and V; the workloads' own queries of sequence 0."""

import os
import sys

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, HERE)
sys.path.insert(0, os.path.dirname(HERE))

import synth  # noqa: E402
from ablation import VARIANTS, attention_rel_err, bytes_per_token_head, rel_err  # noqa: E402


def main():
    n_tok = int(sys.argv[1]) if len(sys.argv) > 1 else 1024
    print("| workload | variant | bytes / token-head | loop error (non-final, mean) | "
          "reference error | attention output error (non-final loops, mean) |")
    print("|---|---|---|---|---|---|")
    for name in ("layer_1p4b", "mixed_24l", "gqa_deep"):
        cfg = synth.config_by_name(name)
        L, d = cfg.n_loops, cfg.head_dim
        rb = list(cfg.res_bits[: L - 1])
        heads = [0, 1]
        x = synth.gen_states(cfg, 0, [0], np.arange(n_tok), heads=heads)[0].astype(np.float64)
        q = synth.gen_queries(cfg, 0, [0])[0].astype(np.float64)     # [Hq][L][d]
        g = cfg.n_q_heads // cfg.n_kv_heads
        signs = synth.rotation_signs(cfg, 0).astype(np.float64)
        for v, f in VARIANTS.items():
            le, re, ae = [], [], []
            for hi, h in enumerate(heads):
                rec = [f(x[:, kv, :, hi, :], signs[h, kv], rb) for kv in range(2)]
                for kv in range(2):
                    e = rel_err(x[:, kv, :, hi, :], rec[kv])
                    le.append(e[: L - 1].mean())
                    re.append(e[L - 1])
                a = attention_rel_err(q[h * g:(h + 1) * g], x[:, 0, :, hi, :],
                                      x[:, 1, :, hi, :], rec[0], rec[1], 1 / np.sqrt(d))
                ae.append(a[: L - 1].mean())
            print("| %s | %s | %d | %.4f | %.4f | %.4f |" % (
                name, v, bytes_per_token_head(v, d, rb), np.mean(le), np.mean(re), np.mean(ae)))


if __name__ == "__main__":
    main()
