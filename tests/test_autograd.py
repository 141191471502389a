"""flash_attn_func, the differentiable form of the forward/backward pair.

CPU: the autograd wiring, with the two kernels' Python entry points replaced
by plain fp64 PyTorch attention so that no GPU is needed -- the gradients
must land on q, k, v in order, and both passes must see the same scale,
mask and dropout arguments.  GPU: with the real kernels, O and the
gradients equal attention_fwd / attention_bwd bit for bit."""
import math

import pytest
import torch

from exact_io_aware_40_gb300 import fa


def _plain(q, k, v, causal, scale):
    s = scale * q @ k.transpose(-1, -2)
    if causal:
        n = q.shape[-2]
        s = s.masked_fill(torch.ones(n, n, dtype=torch.bool).triu(1), float("-inf"))
    return torch.softmax(s, -1) @ v, torch.logsumexp(s, -1)


def test_autograd_wiring_on_cpu(monkeypatch):
    calls = []

    def fake_fwd(q, k, v, causal=False, scale=None, kv_len=None, window=-1, block_mask=None,
                 dropout_p=0.0, seed=0):
        calls.append(("fwd", causal, scale, kv_len, window, block_mask, dropout_p, seed))
        with torch.no_grad():
            return _plain(q, k, v, causal, scale)

    def fake_bwd(q, k, v, o, do, L, causal=False, scale=None, kv_len=None, window=-1,
                 block_mask=None, dropout_p=0.0, seed=0):
        calls.append(("bwd", causal, scale, kv_len, window, block_mask, dropout_p, seed))
        qq, kk, vv = (t.detach().clone().requires_grad_(True) for t in (q, k, v))
        with torch.enable_grad():
            out, _ = _plain(qq, kk, vv, causal, scale)
            return torch.autograd.grad(out, (qq, kk, vv), do)

    monkeypatch.setattr(fa, "attention_fwd", fake_fwd)
    monkeypatch.setattr(fa, "attention_bwd", fake_bwd)
    g = torch.Generator().manual_seed(7)
    q, k, v = (torch.randn(2, 3, 5, 8, generator=g, dtype=torch.float64, requires_grad=True)
               for _ in range(3))
    w = torch.randn(2, 3, 5, 8, generator=g, dtype=torch.float64)

    o, L = fa.flash_attn_func(q, k, v, causal=True, window=4, dropout_p=0.25, seed=11,
                              return_lse=True)
    (o * w).sum().backward()

    ref_q, ref_k, ref_v = (t.detach().clone().requires_grad_(True) for t in (q, k, v))
    ref_o, ref_L = _plain(ref_q, ref_k, ref_v, True, 1 / math.sqrt(8))
    (ref_o * w).sum().backward()
    assert torch.allclose(o, ref_o) and torch.allclose(L, ref_L)
    assert not L.requires_grad
    for got, want in ((q.grad, ref_q.grad), (k.grad, ref_k.grad), (v.grad, ref_v.grad)):
        assert torch.allclose(got, want, rtol=1e-12, atol=1e-12)
    # both passes saw the resolved scale and the same mask / dropout arguments
    assert [c[0] for c in calls] == ["fwd", "bwd"]
    assert calls[0][1:] == calls[1][1:] == (True, 1 / math.sqrt(8), None, 4, None, 0.25, 11)


def test_flash_attn_func_refuses_host_tensors():
    q = torch.zeros(1, 1, 128, 64, dtype=torch.bfloat16, requires_grad=True)
    with pytest.raises(ValueError, match="CUDA"):
        fa.flash_attn_func(q, q, q)


@pytest.mark.gpu
@pytest.mark.parametrize("causal", [False, True])
def test_flash_attn_func_matches_the_kernels(causal):
    from helpers import Case
    case = Case(1701, 2, 3, 300, 64)
    q0, k0, v0, do = (case.dev[n] for n in ("Q", "K", "V", "dO"))
    o_ref, L_ref = fa.attention_fwd(q0, k0, v0, causal=causal, scale=case.scale)
    g_ref = fa.attention_bwd(q0, k0, v0, o_ref, do, L_ref, causal=causal, scale=case.scale)
    q, k, v = (t.detach().clone().requires_grad_(True) for t in (q0, k0, v0))
    o = fa.flash_attn_func(q, k, v, causal=causal, softmax_scale=case.scale)
    o.backward(do)
    fa.fa_check_error()
    assert torch.equal(o, o_ref)
    for got, want in zip((q.grad, k.grad, v.grad), g_ref):
        assert torch.equal(got, want)
