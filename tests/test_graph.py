"""The forward and the backward inside CUDA graphs.

fa_fwd and fa_bwd make no synchronising or allocating CUDA call, so torch's
stream capture records their launches; a replay after new inputs have been
copied into the captured buffers must give bit for bit what direct calls give.
"""
import pytest
import torch

import exact_attention_32_gb300 as fa
from exact_attention_32_gb300 import make_inputs
from exact_attention_32_gb300.workloads import make_grad_output


@pytest.mark.gpu
@pytest.mark.parametrize("B,H,N,d,causal", [(1, 1, 256, 64, False), (2, 4, 1000, 128, True)])
def test_forward_graph_replay_matches_direct_calls(B, H, N, d, causal):
    dev = torch.device("cuda")
    q, k, v = (t.to(dev) for t in make_inputs(B, H, N, d, seed=31))
    o = torch.empty_like(q)
    lse = torch.empty((B, H, N), dtype=torch.float32, device=dev)
    fa.forward(q, k, v, causal=causal, out=o, lse=lse)  # warm-up outside the capture
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        fa.forward(q, k, v, causal=causal, out=o, lse=lse)
    for seed in (32, 33, 34):
        qn, kn, vn = (t.to(dev) for t in make_inputs(B, H, N, d, seed=seed))
        q.copy_(qn)
        k.copy_(kn)
        v.copy_(vn)
        g.replay()
        o_ref, lse_ref = fa.forward(qn, kn, vn, causal=causal)
        torch.cuda.synchronize()
        assert fa.fa_get_device_status(0) == 0
        assert torch.equal(o, o_ref) and torch.equal(lse, lse_ref)


@pytest.mark.gpu
def test_backward_graph_replay_matches_direct_calls():
    dev = torch.device("cuda")
    B, H, N, d = 1, 4, 640, 128
    q, k, v = (t.to(dev) for t in make_inputs(B, H, N, d, seed=41))
    do = make_grad_output(B, H, N, d, 41, device=dev)
    o, lse = fa.forward(q, k, v, causal=True)
    ws = torch.empty(fa.fa_bwd_workspace_bytes(B, H, N, d), dtype=torch.uint8, device=dev)
    dq, dk, dv = (torch.empty_like(q) for _ in range(3))
    s = torch.cuda.Stream()

    def call():
        st = fa.fa_bwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(), do.data_ptr(),
                       dq.data_ptr(), dk.data_ptr(), dv.data_ptr(), B, H, N, d, fa.default_scale(d), True,
                       ws.data_ptr(), ws.numel(), torch.cuda.current_stream().cuda_stream)
        assert st == 0

    call()
    torch.cuda.synchronize()
    ref = [t.clone() for t in (dq, dk, dv)]
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        call()
    for t in (dq, dk, dv):
        t.zero_()
    g.replay()
    torch.cuda.synchronize()
    assert fa.fa_get_device_status(0) == 0
    for t, r in zip((dq, dk, dv), ref):
        assert torch.equal(t, r)
