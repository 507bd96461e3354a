"""Loaders for the hand-derived fixtures under tests/golden/ (inputs + expected values)."""
import json
import os

import numpy as np

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _load(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


def _index(spec, K):
    if isinstance(spec, str) and spec == "all":
        return slice(0, K)
    if isinstance(spec, str):
        a, b = spec.split(":")
        return slice(int(a), int(b))
    return spec


def quant_tie_rule():
    d = _load("quant_tie_rule.json")
    K = d["K"]
    rows = len(d["x_rows_nonzero"])
    x = np.zeros((rows, K), np.float32)
    a_q = np.zeros((rows, K), np.int8)
    for r, items in enumerate(d["x_rows_nonzero"]):
        for k, v in items:
            x[r, k] = np.float32(v)
    for r, items in enumerate(d["expected_a_q_nonzero"]):
        for k, v in items:
            a_q[r, k] = v
    s_a = np.array(d["expected_s_a"], np.float32)
    rs = np.array(d["expected_rowsum"], np.int32)
    return x, a_q, s_a, rs


def linear_hand_cases():
    d = _load("linear_hand_cases.json")
    out = []
    for c in d["cases"]:
        M, K, N = c["M"], c["K"], c["N"]
        x = np.zeros((M, K), np.float32)
        for m, k, v in c["x_nonzero"]:
            x[m, _index(k, K)] = np.float32(v)
        q = np.zeros((N, K), np.uint8)
        for n, k, v in c["q_nonzero"]:
            q[n, _index(k, K)] = v
        wq = (q[:, 0::2] & 0xF) | ((q[:, 1::2] & 0xF) << 4)
        s_w = np.array(c["s_w_fp16_bits"], np.uint16).view(np.float16)
        z_w = np.array(c["z_w_fp16_bits"], np.uint16).view(np.float16)
        bias = None if c["bias"] is None else np.array(c["bias"], np.float32)
        out.append(dict(name=c["name"], x=x, q=q, wq=wq.astype(np.uint8), s_w=s_w, z_w=z_w,
                        bias=bias, y=np.array(c["expected_y"], np.float64)))
    return out
