"""GPU parity of hla_attention_prefill (causal NoPE softmax attention with the
logit scale log_a(p + 1 + a), output norm and gate; arXiv 2601.22156,
Section 5.1 Eq. 11 and Appendix A Eq. 17) against the fp64 oracle."""
import numpy as np
import pytest
import torch

import oracle
from rnn_sequence_mixer_gb300 import api, inputs, workloads
from parity_util import f64, max_rel_err

pytestmark = pytest.mark.gpu

TOL = 2e-2  # bf16 inputs and outputs


@pytest.fixture(scope="module")
def dev():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    return torch.device("cuda:0")


def draw(B, T, Hq, Hkv, seed, dev):
    """q, k, v, gate: N(0, 1) drawn in that order, rounded to bf16."""
    x = inputs.mixer_inputs(B, T, Hq, 128, torch.bfloat16, seed, device=dev)
    kv = inputs.mixer_inputs(B, T, Hkv, 128, torch.bfloat16, seed + 1, device=dev)
    return x["q"], kv["k"], kv["v"], x["gate"]


# (B, T, Hq, Hkv, a, pos_offset): one token, one exact tile, ragged tails over
# several tiles, grouped heads 2:1 and 4:1, a large position offset
CASES = [
    (1, 1, 2, 1, 500.0, 0),
    (1, 128, 2, 2, 500.0, 0),
    (2, 300, 4, 2, 600.0, 7),
    (1, 1000, 4, 1, 900.0, 100000),
    (3, 257, 2, 2, 500.0, 0),
    (1, 129, 8, 2, 600.0, 3),
]


@pytest.mark.parametrize("B,T,Hq,Hkv,a,pos", CASES)
def test_attention_small(dev, B, T, Hq, Hkv, a, pos):
    q, k, v, g = draw(B, T, Hq, Hkv, 40 + T, dev)
    shape = api.make_attn_shape(B, T, Hq, Hkv, 128, a=a, pos_offset=pos)
    ws = torch.full((api.attention_workspace_size(shape),), 0xAB, dtype=torch.uint8, device=dev)
    y, o = api.attention_prefill(q, k, v, g, a, pos_offset=pos, want_o=True, workspace=ws)
    torch.cuda.synchronize()
    assert ws[:4].view(torch.int32).item() == 0
    ry, ro = oracle.attention(f64(q), f64(k), f64(v), f64(g), a, pos_offset=pos)
    assert max_rel_err(f64(o), ro) <= TOL, max_rel_err(f64(o), ro)
    assert max_rel_err(f64(y), ry) <= TOL, max_rel_err(f64(y), ry)


def test_attention_large_logits(dev):
    """q and k scaled by 8: logits of tens, so the running maximum and the
    rescaling of O do real work."""
    B, T, Hq, Hkv, a = 1, 700, 2, 1, 500.0
    q, k, v, g = draw(B, T, Hq, Hkv, 77, dev)
    q, k = (q.float() * 8).to(torch.bfloat16), (k.float() * 8).to(torch.bfloat16)
    y, o = api.attention_prefill(q, k, v, g, a, want_o=True)
    torch.cuda.synchronize()
    ry, ro = oracle.attention(f64(q), f64(k), f64(v), f64(g), a)
    assert torch.isfinite(o).all()
    assert max_rel_err(f64(o), ro) <= TOL
    assert max_rel_err(f64(y), ry) <= TOL


@pytest.mark.parametrize("B,T", [(2, 0), (0, 5)])
def test_attention_empty(dev, B, T):
    q, k, v, g = draw(B, T, 2, 1, 3, dev)
    y, _ = api.attention_prefill(q, k, v, g, 500.0)
    torch.cuda.synchronize()
    assert y.numel() == 0


def test_attention_workload_sampled(dev):
    """B=1, T=16384, Hq=16 over Hkv=8 (the bench's attention workload): two
    query heads of different key/value groups, every token, against the oracle."""
    w = workloads.ATTENTION_16K
    q, k, v, g = draw(w.B, w.T, w.Hq, w.Hkv, w.seed, dev)
    y, o = api.attention_prefill(q, k, v, g, w.a, want_o=True)
    torch.cuda.synchronize()
    for h in (0, 13):
        hk = h // (w.Hq // w.Hkv)
        sel = lambda t, j: f64(t[:, :, j:j + 1, :])
        ry, ro = oracle.attention(sel(q, h), sel(k, hk), sel(v, hk), sel(g, h), w.a)
        assert max_rel_err(sel(o, h), ro) <= TOL
        assert max_rel_err(sel(y, h), ry) <= TOL
