"""Golden values printed on the pages (tests/golden/*.txt, each file cites its
page and section), checked against the oracle.  CPU only."""
import math
import os

import numpy as np
import torch

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _read(name):
    vals = {}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            k, v = (x.strip() for x in line.split("=", 1))
            vals[k] = v
    return vals


def _bits(a):
    return oracle.bf16_bits(torch.tensor(np.asarray(a, np.float32)).to(torch.bfloat16))


def _single_token_score(q, k):
    """lse of a one-token sequence with scale 1 is exactly q . k."""
    d = len(q)
    kv = np.zeros((1, 4, d), np.float32)
    kv[0, 0] = k
    p = oracle.Problem(_bits(np.asarray(q, np.float32).reshape(1, 1, 1, d)), _bits(kv),
                       np.zeros((1, 1), np.int32), np.array([1], np.int32), 1.0, False)
    out, lse = oracle.mla_decode(p, dv=d)
    assert np.array_equal(out[0, 0, 0], np.asarray(k, np.float64))
    return lse[0, 0, 0]


def test_multirail_worked_example():
    g = _read("multirail_dot_example.txt")
    q = [float(x) for x in g["q"].split()]
    k1 = [float(x) for x in g["k1"].split()]
    k2 = [float(x) for x in g["k2"].split()]
    assert _single_token_score(q, k1) == float(g["score_k1"])
    assert _single_token_score(q, k2) == float(g["score_k2"])
    h0 = [float(x) for x in g["half0_partials"].split()]
    h1 = [float(x) for x in g["half1_partials"].split()]
    assert [_single_token_score(q[:2], k[:2]) for k in (k1, k2)] == h0
    assert [_single_token_score(q[2:], k[2:]) for k in (k1, k2)] == h1
    # both tokens: lse = log(e^70 + e^10)
    kv = np.zeros((1, 4, 4), np.float32)
    kv[0, 0], kv[0, 1] = k1, k2
    p = oracle.Problem(_bits(np.asarray(q, np.float32).reshape(1, 1, 1, 4)), _bits(kv),
                       np.zeros((1, 1), np.int32), np.array([2], np.int32), 1.0, False)
    out, lse = oracle.mla_decode(p, dv=4)
    s1, s2 = float(g["score_k1"]), float(g["score_k2"])
    assert abs(lse[0, 0, 0] - (s1 + math.log1p(math.exp(s2 - s1)))) < 1e-12


def test_online_softmax_rescale_example():
    g = _read("online_softmax_rescale_example.txt")
    m_old, m_new = float(g["m_old"]), float(g["m_new"])
    assert g["factor"] == "exp(-2)" and m_old - m_new == -2
    # old state (m=3, l=1, o~=[1]) merged with a fresh block (m=5, l=1, o~=[0]):
    # the old terms are scaled by e^(3-5), the new ones by 1.
    m, l, o = oracle.merge_pair((m_old, 1.0, np.array([1.0])), (m_new, 1.0, np.array([0.0])))
    assert m == m_new
    assert abs(o[0] - math.exp(-2.0)) < 1e-15
    assert abs(l - (math.exp(-2.0) + 1.0)) < 1e-15
