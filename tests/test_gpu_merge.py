"""kvq_merge_splits against the oracle's log-sum-exp merge."""
import numpy as np
import pytest
import torch

import oracle
import quantized_kv_cache_q4_gb300 as kvq
import workloads
from gpu_helpers import dev
from helpers import check_close

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("n_splits,rows,D", [(1, 5, 256), (2, 24, 256), (7, 3, 128), (64, 24, 256),
                                             (256, 24, 256), (1000, 2, 64), (4096, 1, 4), (3, 9, 1024)])
def test_merge_matches_oracle(n_splits, rows, D):
    po, pl = workloads.rand_partials(n_splits, rows, D, seed=n_splits + rows + D)
    pl[:, 0] = -np.inf                    # a row with every part empty
    po[:, 0] = 0
    out = torch.empty((rows, D), dtype=torch.float32, device="cuda")
    lse = torch.empty((rows,), dtype=torch.float32, device="cuda")
    kvq.kvq_merge_splits(dev(po), dev(pl), n_splits, rows, D, out, lse)
    torch.cuda.synchronize()
    o_ref, l_ref = oracle.merge_splits(po, pl)
    check_close(out.cpu().numpy(), o_ref, lse.cpu().numpy(), l_ref, atol=1e-5, rtol_l2=1e-5, lse_atol=1e-5)
    assert np.all(out.cpu().numpy()[0] == 0) and np.isneginf(lse.cpu().numpy()[0])


def test_merge_ignores_values_of_empty_parts():
    po, pl = workloads.rand_partials(8, 4, 256, seed=99, empty_frac=0.0)
    pl[3] = -np.inf
    po[3] = np.nan                        # must never be read
    out = torch.empty((4, 256), dtype=torch.float32, device="cuda")
    kvq.kvq_merge_splits(dev(po), dev(pl), 8, 4, 256, out, None)
    torch.cuda.synchronize()
    po[3] = 0
    o_ref, _ = oracle.merge_splits(po, pl)
    check_close(out.cpu().numpy(), o_ref, atol=1e-5, rtol_l2=1e-5)
