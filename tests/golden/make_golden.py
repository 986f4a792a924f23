"""Writes the golden fixtures of this folder from closed forms.

Uses only the Python standard library (``math``): no oracle and no CUDA code
is involved, so the stored values are independent of both implementations.
Run from the repository root:  python tests/golden/make_golden.py
"""
import json
import math
import os

HERE = os.path.dirname(os.path.abspath(__file__))


def softmax_attention(q, keys, values, scale):
    """Closed-form softmax attention of one query over a few keys (pure math)."""
    s = [scale * sum(a * b for a, b in zip(q, k)) for k in keys]
    m = max(s)
    w = [math.exp(x - m) for x in s]
    z = sum(w)
    return [sum(w[t] * values[t][d] for t in range(len(keys))) / z for d in range(len(values[0]))]


def closed_form_cases():
    # Every number below is exactly representable in bf16.
    q = [1.0, 0.0, 0.0, 0.0]
    k = [[0.0, 0.0, 0.0, 0.0], [2.0, 0.0, 0.0, 0.0]]
    v = [[1.0, 0.0, -1.0, 0.5], [0.0, 1.0, 3.0, -2.0]]
    e = math.e
    # scores (0, 1): weights 1/(1+e) and e/(1+e)
    two = [v[0][d] / (1 + e) + v[1][d] * e / (1 + e) for d in range(4)]
    assert all(abs(a - b) < 1e-15 for a, b in zip(two, softmax_attention(q, k, v, 0.5)))

    q3 = [1.0, 1.0, 0.0, -0.5]
    k3 = [[1.0, 0.0, 0.0, 0.0], [0.0, 1.0, 0.0, 0.0], [1.0, 1.0, 0.0, 2.0]]
    v3 = [[0.5, -1.0, 2.0, 0.0], [1.5, 0.25, -3.0, 1.0], [-2.0, 4.0, 0.125, -0.75]]
    # verify block of two new rows (q_len 2) over a 3-token context: row 0 sees
    # keys 0..1, row 1 sees keys 0..2
    qa = [0.5, -1.0, 0.0, 1.0]
    return {
        "citation": ("Closed-form softmax attention, the plain definition the pages' kernels compute: "
                     "'DCU page832 attention' Sec.5 (score = dot(Q, K) * scale, online softmax "
                     "over the keys); verify rows with a per-row causal mask: 'Qwen3.8 on MI350P' "
                     "Lektion 3."),
        "cases": [
            {"name": "two_tokens", "head_dim": 4, "scale": 0.5, "q_len": 1, "q": [q], "k": k, "v": v,
             "expected": [two],
             "derivation": "scores (0, 1); out = V0/(1+e) + V1*e/(1+e)"},
            {"name": "three_tokens", "head_dim": 4, "scale": 0.25, "q_len": 1, "q": [q3], "k": k3, "v": v3,
             "expected": [softmax_attention(q3, k3, v3, 0.25)],
             "derivation": "scores 0.25*(1, 1, 1); equal weights -> mean of V"},
            {"name": "verify_two_rows", "head_dim": 4, "scale": 0.5, "q_len": 2, "q": [qa, q3],
             "k": k3, "v": v3,
             "expected": [softmax_attention(qa, k3[:2], v3[:2], 0.5),
                          softmax_attention(q3, k3, v3, 0.5)],
             "derivation": "row r of a q_len block sees keys 0 .. L - q_len + r"},
        ],
    }


def address_cases():
    rows = []
    for bs, t in [(784, 783), (784, 784), (784, 800), (784, 32767), (832, 831), (832, 832),
                  (832, 8207), (16, 0), (16, 511)]:
        rows.append({"block_size": bs, "token": t, "logical_page": t // bs, "page_offset": t % bs})
    return {
        "citation": ("'DCU page832 attention' Sec.1: logical_page = token // BLOCK_SIZE, "
                     "page_offset = token % BLOCK_SIZE, physical_page = block_table[logical_page]; "
                     "Sec.2: 784 = 12 x 64 + 16 and 832 = 13 x 64."),
        "page_tiling": [{"block_size": 784, "full_64_tiles": 12, "tail_tokens": 16},
                        {"block_size": 832, "full_64_tiles": 13, "tail_tokens": 0}],
        "examples": rows,
    }


if __name__ == "__main__":
    with open(os.path.join(HERE, "closed_form_attention.json"), "w") as f:
        json.dump(closed_form_cases(), f, indent=1)
    with open(os.path.join(HERE, "page_address.json"), "w") as f:
        json.dump(address_cases(), f, indent=1)
    print("written")
