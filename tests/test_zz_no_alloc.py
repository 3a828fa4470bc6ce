"""The allocation-free attention entry point (dsa_sparse_mla_fwd_noalloc),
called through the C ABI, against the workspace entry point on the same
inputs, two calls in a row.

It serves callers that cannot allocate device memory where attention runs
(a serving loop under a fixed memory plan, or an embedder without access to
the allocator): its split-K partials live in the library's static device
scratch instead of a caller-provided workspace.  This file is collected last
on purpose.
"""

import ctypes

import numpy as np
import pytest
import torch

import sparse_attention_gb300 as dsa
import workloads as W
from dsa_case import ATT_ATOL, ATT_RTOL, Staged

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lib():
    from sparse_attention_gb300 import build as B
    B.build()
    return dsa.load_library()


def _case(seed):
    # few query rows, so each row's selected list is split over several CTAs
    # and the split-K partials go through the scratch
    bt = W.make_batch_np([1000, 2500, 128, 4097, 3000], [1, 1, 1, 1, 1], k=2048, seed=seed, key_kind="zipf")
    st = Staged(bt)
    ix = st.topk(st.scores())
    return st, ix


def _noalloc(lib, st, ix, out, lse, status):
    rc = lib.dsa_sparse_mla_fwd_noalloc(ctypes.byref(st.b.c), st.q.data_ptr(), st.kv.data_ptr(), ix.data_ptr(),
                                        st.bt.k, ctypes.c_float(st.bt.sm_scale), out.data_ptr(), lse.data_ptr(),
                                        status.data_ptr(), ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert rc == 0, dsa.STATUS.get(rc, rc)


def test_noalloc_matches_workspace_entry_point_twice(lib):
    for call, seed in enumerate((501, 502)):
        st, ix = _case(seed)
        ref_out, ref_lse = st.attention(ix)
        out = torch.full_like(ref_out, float("nan"))
        lse = torch.full_like(ref_lse, float("nan"))
        status = torch.zeros(1, dtype=torch.int32, device="cuda")
        _noalloc(lib, st, ix, out, lse, status)
        torch.cuda.synchronize()
        assert int(status.item()) == 0
        r, o = ref_out.float().cpu().numpy(), out.float().cpu().numpy()
        assert np.all(np.abs(o - r) <= ATT_ATOL + ATT_RTOL * np.abs(r)), f"call {call}: output differs"
        rl, ol = ref_lse.cpu().numpy(), lse.cpu().numpy()
        assert np.allclose(ol, rl, rtol=1e-3, atol=1e-3), f"call {call}: lse differs"
        # same kernels and the same split of each row: the same bits
        assert torch.equal(out.view(torch.int16), ref_out.view(torch.int16))



def test_noalloc_rejects_partials_beyond_the_static_array(lib):
    # 100 query rows at k = 2047 split each row in three (merged by a second
    # kernel, not in a cluster): 300 partials of 131,328 B do not fit in
    # 32 MiB.  Every buffer is real and sized for the batch (all indices -1),
    # so the call could not touch memory it does not own even if it
    # launched; it must refuse before launching.
    T, ctx, k = 100, 4096, 2047
    b = dsa.make_batch([0, T], [ctx], T, ctx, ctx)
    q = torch.zeros((T, 64, 576), dtype=torch.bfloat16, device="cuda")
    kv = torch.zeros((ctx, 576), dtype=torch.bfloat16, device="cuda")
    ix = torch.full((T, k), -1, dtype=torch.int32, device="cuda")
    out = torch.zeros((T, 64, 512), dtype=torch.bfloat16, device="cuda")
    n0 = dsa.kernel_launch_count()
    rc = lib.dsa_sparse_mla_fwd_noalloc(ctypes.byref(b.c), q.data_ptr(), kv.data_ptr(), ix.data_ptr(), k,
                                        ctypes.c_float(0.0625), out.data_ptr(), None, None, None)
    assert rc == 3          # DSA_ERR_WORKSPACE
    assert dsa.kernel_launch_count() == n0
