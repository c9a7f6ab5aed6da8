"""Write the oracle's full-size forward results for the large workloads.

Calls only ``oracle`` (and the seeded input generator).  For each workload it
stores the loss, N_valid and the per-row lse (fp64) so that GPU tests at full
size can compare lse and the loss directly and rebuild dz columns for sampled
dW rows without a full fp64 forward on the GPU host.

    python tests/golden/make_golden.py 1 2 3 4
"""
import os
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
sys.path.insert(0, ROOT)

import oracle  # noqa: E402
from lm_head_kl_fkl_b300 import synth  # noqa: E402

HERE = os.path.dirname(os.path.abspath(__file__))


def golden_path(i):
    return os.path.join(HERE, f"oracle_forward_cfg{i}.npz")


def main(which):
    for i in which:
        t0 = time.time()
        x = synth.config_inputs(i)
        h = synth.bf16_bits_to_f64(x["h"])
        W = synth.bf16_bits_to_f64(x["W"])
        out = oracle.forward(h, W, x["idx"], x["t"], x["mask"], x["T"], row_block=256)
        np.savez(golden_path(i), loss=np.float64(out["loss"]), lse=out["lse"],
                 n_valid=np.int64(out["n_valid"]), fingerprint=np.str_(synth.fingerprint(x)),
                 name=np.str_(x["name"]))
        print(f"cfg{i} {x['name']}: loss={out['loss']:.12g} n_valid={out['n_valid']} "
              f"({time.time() - t0:.0f} s)", flush=True)


if __name__ == "__main__":
    main([int(a) for a in sys.argv[1:]] or [1, 2, 3, 4])
