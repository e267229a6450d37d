"""Writes synth/zipf_bias_beta.json: the strength beta of the Zipf-shaped correction
bias of the skewed-routing workload (T=16384, H=7168, E=384, top-8), found by
bisection with the oracle's router so that the most popular expert receives
8.0% +- 0.2% of the routed assignments.

The bias is  bias_e = beta * (-1.1 * ln rank_e)  with rank a seeded
permutation of the experts (synth.zipf_ranks).  Pure Zipf(1.1) over 384 ranks
would put 19.7% of the mass on rank 1, but distinct top-8 routing caps any
expert at 12.5% of assignments; the workload asks for ~8%, so the bias keeps
the Zipf shape and beta sets the strength.

Run:  python tests/golden/make_zipf_beta.py      (uses only oracle/ and synth)
"""
import json
import sys
from dataclasses import replace
from pathlib import Path

import numpy as np

ROOT = Path(__file__).resolve().parents[2]
sys.path.insert(0, str(ROOT))

import synth  # noqa: E402
from oracle.router import route, router_logits  # noqa: E402


def hottest_share(cfg, logits, beta):
    bias = synth.gen_bias_f32(cfg, beta=beta)
    idx, _ = route(logits, bias, cfg.top_k, cfg.n_group, cfg.topk_group, cfg.routed_scaling,
                   cfg.renormalize)
    counts = np.bincount(idx.reshape(-1), minlength=cfg.E)
    return counts.max() / idx.size, counts


def main():
    cfg = synth.configs()["skewed_shared"]
    x = synth.bf16_bits_to_f64(synth.gen_x_bf16(cfg))
    wr = synth.bf16_bits_to_f64(synth.gen_router_bf16(cfg))
    logits, _ = router_logits(x, wr)
    lo, hi = 0.0, 4.0
    for _ in range(40):
        mid = 0.5 * (lo + hi)
        share, _ = hottest_share(cfg, logits, mid)
        if share < 0.08:
            lo = mid
        else:
            hi = mid
        if abs(share - 0.08) < 0.0005:
            break
    beta = mid
    share, counts = hottest_share(cfg, logits, beta)
    top = np.sort(counts)[::-1]
    out = {"beta": beta, "hottest_share": float(share),
           "share_curve_top16": [float(c / (cfg.T * cfg.top_k)) for c in top[:16]],
           "touched_experts": int(np.count_nonzero(counts)),
           "note": "written by tests/golden/make_zipf_beta.py with the oracle router"}
    (ROOT / "synth" / "zipf_bias_beta.json").write_text(json.dumps(out, indent=1) + "\n")
    print(json.dumps(out))


if __name__ == "__main__":
    main()
