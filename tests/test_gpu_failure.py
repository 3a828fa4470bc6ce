"""Failure detection without a GPU fault: a kernel's bounded wait on a
barrier that nothing completes must give up, latch DSA_ERR_TIMEOUT in the
workspace status word and return, leaving the context usable."""

import numpy as np
import pytest
import torch

import sparse_attention_gb300 as dsa
import workloads as W
from dsa_case import Staged, check_attention

pytestmark = pytest.mark.gpu


def test_bounded_wait_latches_timeout_and_context_survives():
    from sparse_attention_gb300 import build as B
    B.build()
    dsa.load_library()
    bt = W.make_batch_np([300], [2], k=64, seed=91)
    st = Staged(bt)
    assert st.status() == 0
    dsa.selftest_wait_timeout(st.ws, limit_us=2000)       # a 2 ms wait that runs out
    assert st.status() == 5                                # DSA_ERR_TIMEOUT
    dsa.reset_device_status(st.ws)
    assert st.status() == 0
    # the context still runs the path correctly
    ix = st.topk(st.scores())
    out, lse = st.attention(ix)
    check_attention(st, ix, out, lse)
    assert st.status() == 0


def test_selftest_rejects_bad_limits():
    ws = torch.zeros(256, dtype=torch.uint8, device="cuda")
    with pytest.raises(dsa.DsaError):
        dsa.selftest_wait_timeout(ws, limit_us=0)
    with pytest.raises(dsa.DsaError):
        dsa.selftest_wait_timeout(ws, limit_us=2_000_000)
