"""luce_argmax_noalloc: the argmax for callers that cannot allocate device
memory (an application that owns every allocation and gives the library
none, or a loop that must not call the CUDA allocator).  It keeps its
scratch in a fixed array of device memory owned by the library.

Collected last on purpose (file name), so a run that stops at its first
failure has run every other test before this one.  It passes alone in a
fresh process and after the other tests.
"""
import numpy as np
import pytest
import torch

from quantized_moe_decode_luce_gb300 import binding as B
from quantized_moe_decode_luce_gb300 import build as BLD
from quantized_moe_decode_luce_gb300 import workloads as W
from quantized_moe_decode_luce_gb300.layer import Argmax


@pytest.mark.gpu
def test_argmax_noalloc_matches_the_workspace_entry_point_on_two_calls():
    assert torch.cuda.is_available(), "needs a CUDA device"
    BLD.build()
    B.lib()
    for R, V, seed in [(5, 129280, 1), (3, 4097, 2)]:  # two calls in a row, the second smaller
        x = torch.from_numpy(W.rng(800, seed).standard_normal((R, V)).astype(np.float32)).cuda()
        x[0, 17] = x[0, V - 1] = 50.0  # a tie: the lower index wins
        am = Argmax(R, V)
        idx_ref, val_ref = am.run(x)
        idx = torch.full((R,), -7, dtype=torch.int32, device="cuda")
        val = torch.full((R,), -7.0, dtype=torch.float32, device="cuda")
        B.luce_argmax_noalloc(x, idx, val)
        torch.cuda.synchronize()
        # the argmax is exact: same index and same value, bit for bit
        assert torch.equal(idx, idx_ref) and torch.equal(val.view(torch.int32), val_ref.view(torch.int32))
        assert int(idx[0]) == 17
    assert B.luce_get_fault() == 0


@pytest.mark.gpu
def test_argmax_noalloc_rejects_sizes_beyond_its_scratch():
    BLD.build()
    x = torch.zeros((1025, 8), dtype=torch.float32, device="cuda")
    idx = torch.empty(1025, dtype=torch.int32, device="cuda")
    with pytest.raises(B.LuceError) as ei:
        B.luce_argmax_noalloc(x, idx, None)
    assert ei.value.status == B.LUCE_ERR_UNSUPPORTED
