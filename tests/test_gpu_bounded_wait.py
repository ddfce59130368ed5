"""The bounded waits' failure path on the GPU, without a fault or a hang: a
wait on an mbarrier that nothing arrives at gives up after a few polls and
records a timeout; csa2_check_device_error reports it once, and the context
stays usable (a scoring call afterwards still matches the oracle)."""
import numpy as np
import pytest
import torch

from gpu_util import assert_scores_close, need_gpu, np_
from oracle import csa2_oracle as o
from serving_lightning_indexer_gb300 import csa2
from serving_lightning_indexer_gb300 import workloads as W

pytestmark = pytest.mark.gpu


def test_a_wait_that_runs_out_returns_the_timeout_status_and_the_context_stays_usable():
    dev = need_gpu()
    lib = csa2.load()
    stream = torch.cuda.current_stream()
    assert csa2.check_device_error() == 0                    # nothing recorded before
    assert lib.csa2_debug_bounded_wait(64, stream.cuda_stream) == 0
    assert csa2.check_device_error() == 8                    # CSA2_ERR_DEVICE_TIMEOUT
    assert b"bounded wait" in lib.csa2_last_error_detail()
    assert csa2.check_device_error() == 0                    # the record was cleared
    assert lib.csa2_debug_bounded_wait(0, stream.cuda_stream) == 2        # polls out of range
    assert lib.csa2_debug_bounded_wait((1 << 20) + 1, stream.cuda_stream) == 2

    # a normal call afterwards: scores of a short row against the oracle
    n = 3000
    pc = W.make_paged_cache([n], seed=40, device=dev, with_main=False)
    iq = W.make_indexer_query(1, seed=41, device=dev)
    scores = torch.empty(1, 3072, dtype=torch.float32, device=dev)
    csa2.index_score(iq.q_fp8, iq.q_scale, iq.w, pc.index_k, pc.page_table, csa2.rows(1, 1, n_visible=pc.n_entries),
                     scores)
    assert csa2.check_device_error() == 0
    ref = o.index_scores_row(np_(iq.q_fp8[0]), np_(iq.q_scale[0]), np_(iq.w[0]), np_(pc.index_k),
                             np_(pc.page_table[0]), n)
    assert_scores_close(np_(scores[0, :n]), ref)
    assert np.isneginf(np_(scores[0, n:])).all()
