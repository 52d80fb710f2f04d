"""Write tests/golden/oracle_small.json: oracle outputs for small seeded inputs.

Calls only the oracle (and numpy's seeded generator for the inputs).  The stored
digests freeze the oracle's readings of the page; a change to the oracle's
arithmetic that alters them must regenerate this file and say why in its commit.
Run:  python tests/golden/make_golden.py
"""
import hashlib
import json
import os
import sys

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(os.path.dirname(HERE)))
import oracle  # noqa: E402


def bf16_bits_from_f32(a: np.ndarray) -> np.ndarray:
    """fp32 -> bf16 bit patterns, round to nearest even (input generator step)."""
    u = a.astype(np.float32).view(np.uint32).astype(np.uint64)
    u = (u + 0x7FFF + ((u >> 16) & 1)) >> 16
    return u.astype(np.uint16)


CASES = [
    # name, shape, std, block, round, rht, sr_seed, rht_seed
    ("row_rne", (32, 64), 1.0, oracle.ROW, oracle.RNE, False, 0, 0),
    ("row_sr", (32, 64), 1e-3, oracle.ROW, oracle.SR, False, 0, 0),
    ("col_rht_sr", (64, 48), 1e-3, oracle.COL, oracle.SR, True, 0, 1),
    ("col_rht_rne", (64, 48), 1.0, oracle.COL, oracle.RNE, True, 0, 1),
    ("tile_rne", (48, 64), 0.02, oracle.TILE16, oracle.RNE, False, 0, 0),
]


def digest(a: np.ndarray) -> str:
    return hashlib.sha256(np.ascontiguousarray(a).tobytes()).hexdigest()


def make():
    out = {"_how": "inputs: numpy default_rng(seed=case index).standard_normal(shape)*std -> bf16 (RNE); "
                   "outputs: oracle.quantize (oracle.mx_quantize for the mx_ cases); digests are sha256 of "
                   "the raw code / scale bytes"}
    for i, (name, shape, std, block, rnd, rht, sr_seed, rht_seed) in enumerate(CASES):
        x = bf16_bits_from_f32(np.random.default_rng(i).standard_normal(shape) * std)
        q = oracle.quantize(x, block, rnd, rht=rht, sr_seed=sr_seed, rht_seed=rht_seed)
        out[name] = dict(shape=list(shape), std=std, block=block, round=rnd, rht=rht,
                         sr_seed=sr_seed, rht_seed=rht_seed, seed=i,
                         s_dec=float(np.float32(q["s_dec"])).hex(),
                         codes_sha256=digest(q["codes"]), scales_sha256=digest(q["scales"]),
                         first_codes=q["codes"][0, :8].tolist(), first_scales=q["scales"][0, :4].tolist())
    # MXFP4 (the comparison format): 1x32 blocks, UE8M0 scales, rows and the transposed operand
    for j, (name, shape, std, col) in enumerate((("mx_row", (32, 96), 1.0, False), ("mx_col", (64, 48), 0.02, True))):
        seed = len(CASES) + j
        x = bf16_bits_from_f32(np.random.default_rng(seed).standard_normal(shape) * std)
        q = oracle.mx_quantize(x, col=col)
        out[name] = dict(shape=list(shape), std=std, col=col, seed=seed,
                         codes_sha256=digest(q["codes"]), scales_sha256=digest(q["scales"]),
                         first_codes=q["codes"][0, :8].tolist(), first_scales=q["scales"][0, :2].tolist())
    return out


if __name__ == "__main__":
    with open(os.path.join(HERE, "oracle_small.json"), "w") as f:
        json.dump(make(), f, indent=1)
    print("wrote oracle_small.json")
