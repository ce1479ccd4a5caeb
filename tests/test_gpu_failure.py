"""Failure detection without a GPU fault: a barrier wait whose partner never
arrives gives up within its budget, reports BSA_ERR_TIMEOUT through the status
word, and the context keeps running the path afterwards."""
import numpy as np
import pytest
import torch

import dynamic_block_sparse_mean_gb300 as bsa
import oracle
from dynamic_block_sparse_mean_gb300 import synth
from parity_utils import BF16_MAX_ABS, oracle_view, shape_of, upload, worklist_from_oracle

pytestmark = pytest.mark.gpu


def test_bounded_wait_times_out_and_context_stays_usable():
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    bsa.selftest_wait_timeout(status)
    torch.cuda.synchronize()
    assert int(status.item()) == 19                     # BSA_ERR_TIMEOUT
    # first error wins: a second run leaves the recorded code alone
    status.fill_(16)
    bsa.selftest_wait_timeout(status)
    torch.cuda.synchronize()
    assert int(status.item()) == 16
    # the context still computes the path
    x = synth.gen_prefill([300], 2, 2, 64, 64, 4, "iid", "bf16")
    q, k, v = upload(x)
    sh = shape_of(x, 2, 2)
    Jo, co, _, _ = oracle.route(oracle_view(x, "q"), oracle_view(x, "k"), x.cu_seqlens, 64, 1,
                                oracle.TOPK, 3)
    ok = torch.zeros(1, dtype=torch.int32, device="cuda")
    wl = worklist_from_oracle(Jo, co, sh, 3, ok)
    O, lse = bsa.attention_fwd(q, k, v, wl, sh, ok)
    torch.cuda.synchronize()
    bsa.check_status(ok)
    Oo, lo = oracle.attention(oracle_view(x, "q"), oracle_view(x, "k"), oracle_view(x, "v"),
                              x.cu_seqlens, 64, 1, Jo, co)
    assert np.abs(O.float().cpu().numpy() - Oo).max() <= BF16_MAX_ABS
