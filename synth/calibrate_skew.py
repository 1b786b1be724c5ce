"""Write ``synth/skew_offsets.json``: router logit offsets c_e that give the
Zipf(1.1)-skewed expert loads of the V4-Pro-shaped workloads.

Run once, offline: ``python synth/calibrate_skew.py``.  The offsets are input
parameters, not expected values.  The fixed point is taken with the oracle's
routing (``oracle.route_from_logits``) on seeded logits l = c_e + z,
z ~ N(0, 1), which is the distribution the workload's X Wg produces when
X[:, 0] = 1 and Wg[0, e] = c_e (the other H-1 terms sum to ~N(0, 1)).
"""
import json
import os
import sys

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(HERE))

import oracle  # noqa: E402
import synth  # noqa: E402


def calibrate(name, seed=1234, reps=2, iters=300):
    cfg = synth.get_config(name)
    T, E, k = cfg["T"], cfg["E"], cfg["k"]
    tgt = synth.zipf_targets(E, T * k, T)
    bias = synth.make_inputs(dict(cfg, T=0, H=64, I=64), seed=seed)["bias"]
    rng = np.random.default_rng(4321)
    z = rng.standard_normal((reps * T, E))
    c = np.log(np.maximum(tgt, 0.5) / tgt.mean())
    for it in range(iters):
        ids, _, _ = oracle.route_from_logits(z + c[None, :], bias, cfg["score_fn"], k,
                                             cfg["alpha"], cfg["renorm"])
        real = np.bincount(ids.reshape(-1), minlength=E) / reps
        tv = 0.5 * np.abs(real - tgt).sum() / tgt.sum()  # total-variation distance
        if tv < 0.01 and it > 5:
            break
        step = 0.4 * (np.log(tgt + 0.5) - np.log(real + 0.5))
        c = np.clip(c + np.clip(step, -0.5, 0.5), -12.0, 12.0)
    c32 = np.asarray(synth.f32_from_bf16_bits(synth.bf16_bits_from_f32(c.astype(np.float32))))
    key = f"E{E}_k{k}_{cfg['score']}_{cfg['skew']}"
    return key, dict(c=[float(v) for v in c32], targets=[float(v) for v in tgt],
                     realized=[float(v) for v in real], tv_distance=float(tv),
                     T=T, seed=seed, iters=it + 1)


if __name__ == "__main__":
    out = {}
    for name in ("c3", "c3s"):
        key, rec = calibrate(name)
        print(name, key, "iters", rec["iters"], "TV", round(rec["tv_distance"], 4),
              "hottest", max(rec["realized"]), "coldest", min(rec["realized"]))
        out[key] = rec
    with open(os.path.join(HERE, "skew_offsets.json"), "w") as f:
        json.dump(out, f, indent=0)
