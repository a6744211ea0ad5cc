"""GPU parity of the sigmoid top-K router and of the routed call.

The router ("MoE Expert Kernels", section 1; the Hy3 decode write-up, the
router after its logits) against its oracle: the selection is an integer
decision taken in float32 on both sides. The GPU's float32 sigmoid (CUDA expf)
and the oracle's (numpy) may differ in the last bit, so where the two
selections differ the GPU's must still be a valid one: its choice scores,
read with the oracle's float32 arithmetic, equal the oracle's to a few ulps
and are in non-increasing order. The weights match to 2e-6 relative.
"""
import numpy as np
import pytest
import torch

from oracle import router as R
from mxfp4_routed_expert_route_gb300 import (device_errors, mxfp4_expert_linear,
                                             mxfp4_expert_linear_routed, router_topk,
                                             wait_timeouts, workloads)
from gpu_util import TOL, assert_parity
import oracle

pytestmark = pytest.mark.gpu


def _logits(rng, T, E):
    return rng.normal(size=(T, E)).astype(np.float32)


def check_router(logits, bias, K, scaling, sel, p):
    sel = sel.cpu().numpy().astype(np.int64)
    p = p.cpu().numpy().astype(np.float64)
    want_sel, want_p = R.router(logits, np.zeros(logits.shape[1]) if bias is None else bias,
                                K, scaling)
    raw, choice = R.choice_scores(logits, np.zeros(logits.shape[1]) if bias is None else bias)
    differ = 0
    for t in range(sel.shape[0]):
        if np.array_equal(sel[t], want_sel[t]):
            np.testing.assert_allclose(p[t], want_p[t], rtol=2e-6, atol=1e-30)
            continue
        differ += 1
        got_c = choice[t, sel[t]].astype(np.float64)
        want_c = choice[t, want_sel[t]].astype(np.float64)
        ulp = np.spacing(np.abs(want_c).astype(np.float32)).astype(np.float64)
        assert np.all(np.abs(got_c - want_c) <= 4 * ulp), (t, sel[t], want_sel[t])
        assert np.all(np.diff(got_c) <= 4 * ulp[1:])
        assert len(set(sel[t].tolist())) == K
        s = raw[t, sel[t]].astype(np.float64)
        np.testing.assert_allclose(p[t], s / (s.sum() + 1e-20) * scaling, rtol=2e-6)
    return differ


@pytest.mark.parametrize("T,E,K", [(8, 128, 4), (16, 384, 8), (4096, 128, 4), (33, 5, 2),
                                   (7, 40, 40), (3, 1000, 1), (2, 2048, 16)])
def test_router_matches_oracle(T, E, K):
    rng = np.random.default_rng(T * 7 + E)
    logits = _logits(rng, T, E)
    bias = rng.normal(0, 0.1, E).astype(np.float32)
    sel, p = router_topk(torch.from_numpy(logits).cuda(), torch.from_numpy(bias).cuda(), K, 2.5)
    torch.cuda.synchronize()
    differ = check_router(logits, bias, K, 2.5, sel, p)
    assert differ <= max(1, T // 100)


def test_router_ties_nan_and_no_bias():
    rng = np.random.default_rng(9)
    T, E, K = 6, 70, 6
    logits = _logits(rng, T, E)
    logits[0] = 0.5                      # every expert ties: 0..5 in order
    logits[1, 10] = logits[1, 3] = 9.0   # a tie at the top: 3 before 10
    logits[2, :] = np.nan
    logits[2, 60:64] = 1.0               # only four valid experts in row 2
    logits[3, ::2] = np.nan
    sel, p = router_topk(torch.from_numpy(logits).cuda(), None, K)
    sel, p = sel.cpu().numpy(), p.cpu().numpy()
    assert sel[0].tolist() == list(range(6))
    assert sel[1, :2].tolist() == [3, 10]
    assert sel[2].tolist() == [60, 61, 62, 63, -1, -1] and (p[2, 4:] == 0).all()
    assert np.allclose(p[2, :4], 0.25)
    assert (sel[3] % 2 == 1).all()
    ok = [0, 1, 4, 5]
    check_router(logits[ok], None, K, 1.0, torch.from_numpy(sel[ok]), torch.from_numpy(p[ok]))


@pytest.mark.parametrize("name", ["decode", "wide_decode", "prefill"])
def test_routed_linear(name):
    # Router, then linear, in one call: the same bits as the two calls, and
    # the oracle composition (oracle router, then oracle linear) within the
    # linear's tolerance.
    rng = np.random.default_rng(len(name))
    wl = workloads.named(name)
    logits = _logits(rng, wl.T, wl.E)
    bias = rng.normal(0, 0.1, wl.E).astype(np.float32)
    d = wl.device_tensors("cuda")
    lg, b = torch.from_numpy(logits).cuda(), torch.from_numpy(bias).cuda()
    out, sel, p = mxfp4_expert_linear_routed(d["x"], d["packed"], d["scales"], lg, b, wl.K,
                                             d["y_shared"], scaling=1.0)
    torch.cuda.synchronize()
    assert wait_timeouts() == 0
    sel2, p2 = router_topk(lg, b, wl.K, 1.0)
    assert torch.equal(sel, sel2) and torch.equal(p, p2)
    ref = mxfp4_expert_linear(d["x"], d["packed"], d["scales"], sel2, p2, d["y_shared"])
    assert torch.equal(out, ref)
    rows = np.array(sorted({0, wl.T // 2, wl.T - 1}))
    check_router(logits[rows], bias, wl.K, 1.0, sel[torch.from_numpy(rows).cuda()],
                 p[torch.from_numpy(rows).cuda()])
    want, absm, _ = oracle.expert_linear(wl.x, wl.packed, wl.scales, sel.cpu().long(),
                                         p.cpu(), wl.y_shared, rows=rows)
    assert_parity(out[torch.from_numpy(rows).cuda()], want, absm, wl.dtype, f"routed {name}")


@pytest.mark.parametrize("T,E,K,dtype", [(8, 128, 4, torch.bfloat16), (16, 384, 8, torch.bfloat16),
                                         (3, 40, 3, torch.float32), (1, 8, 8, torch.bfloat16),
                                         (200, 64, 5, torch.bfloat16)])
def test_routed_call_matches_router_then_linear(T, E, K, dtype):
    # Ties within a token and a scaling factor: the routed call gives the
    # same bits as the router, then the linear on its output.
    wl = workloads.make(T, E, K, 320, 96, dtype=dtype, seed=T + E)
    rng = np.random.default_rng(T * E)
    logits = _logits(rng, T, E)
    logits[0, :4] = logits[0, 4]
    bias = rng.normal(0, 0.1, E).astype(np.float32)
    d = wl.device_tensors("cuda")
    lg, b = torch.from_numpy(logits).cuda(), torch.from_numpy(bias).cuda()
    out, sel, p = mxfp4_expert_linear_routed(d["x"], d["packed"], d["scales"], lg, b, K,
                                             d["y_shared"], scaling=2.5)
    sel2, p2 = router_topk(lg, b, K, 2.5)
    out2 = mxfp4_expert_linear(d["x"], d["packed"], d["scales"], sel2, p2, d["y_shared"])
    torch.cuda.synchronize()
    assert wait_timeouts() == 0
    assert torch.equal(sel, sel2) and torch.equal(p, p2) and torch.equal(out, out2)
    check_router(logits, bias, K, 2.5, sel, p)


def test_routed_call_with_nan_logits():
    # A token whose logits are all NaN gets no expert: ids -1, weights 0,
    # counted as invalid pairs, and its output is the shared output.
    wl = workloads.make(4, 16, 2, 64, 40, dtype=torch.float32, seed=5)
    logits = np.random.default_rng(3).standard_normal((4, 16)).astype(np.float32)
    logits[2, :] = np.nan
    d = wl.device_tensors("cuda")
    device_errors()
    out, sel, p = mxfp4_expert_linear_routed(d["x"], d["packed"], d["scales"],
                                             torch.from_numpy(logits).cuda(), None, 2,
                                             d["y_shared"])
    torch.cuda.synchronize()
    assert sel[2].tolist() == [-1, -1] and p[2].tolist() == [0.0, 0.0]
    assert device_errors() == 2
    assert torch.equal(out[2].cpu(), wl.y_shared[2])
