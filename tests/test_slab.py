"""fa_fwd_slab on one GPU: the slabs of every rank of a world, run one after
the other on the same tensors, write exactly the rows of their own (b, h)
slices, and together give fa_fwd's result bit for bit (the same kernel runs
on each slab as a problem of its own, and the slices are independent)."""
import numpy as np
import pytest
import torch

import exact_attention_32_gb300 as fa
from exact_attention_32_gb300 import make_inputs

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("B,H,N,d,causal,world", [(2, 3, 300, 128, True, 4), (1, 5, 1000, 64, False, 3),
                                                 (1, 2, 257, 64, True, 3)])
def test_slabs_of_all_ranks_equal_the_whole_forward(B, H, N, d, causal, world):
    q, k, v = (t.cuda() for t in make_inputs(B, H, N, d, seed=40 + world + d))
    scale = fa.default_scale(d)
    o_ref, lse_ref = fa.forward(q, k, v, scale=scale, causal=causal)
    o = torch.full_like(q, float("nan"))
    lse = torch.full((B, H, N), float("nan"), device="cuda")
    stream = torch.cuda.current_stream().cuda_stream
    for rank in range(world):
        begin, count = fa.fa_bh_partition(B * H, world, rank)
        st = fa.fa_fwd_slab(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(),
                            B, H, N, d, scale, causal, rank, world, stream)
        assert st == 0, fa.fa_status_string(st)
        torch.cuda.synchronize()
        written = ~torch.isnan(lse.reshape(-1, N)).all(dim=1)
        # after rank r, exactly the slices of ranks 0..r are written
        assert written.nonzero().flatten().tolist() == list(range(begin + count))
    assert fa.fa_get_device_status(0) == 0
    assert torch.equal(o, o_ref) and torch.equal(lse, lse_ref)


def test_empty_slab_launches_nothing():
    q = torch.zeros((1, 1, 128, 64), dtype=torch.bfloat16, device="cuda")
    o = torch.full_like(q, 7.0)
    lse = torch.full((1, 1, 128), 7.0, device="cuda")
    st = fa.fa_fwd_slab(q.data_ptr(), q.data_ptr(), q.data_ptr(), o.data_ptr(), lse.data_ptr(),
                        1, 1, 128, 64, 0.125, 0, 1, 2, None)
    assert st == 0
    torch.cuda.synchronize()
    assert bool((o == 7.0).all()) and bool((lse == 7.0).all())
    assert fa.fa_fwd_slab(q.data_ptr(), q.data_ptr(), q.data_ptr(), o.data_ptr(), lse.data_ptr(),
                          1, 1, 128, 64, 0.125, 0, 2, 2, None) == 1
