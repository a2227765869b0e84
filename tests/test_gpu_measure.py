"""The measurement reference sdm_measure_row_traffic (the scan's row traffic
with no arithmetic): every piece it writes is a whole, unaltered piece of the
same chain and columns of the source table, and it writes nothing else."""
import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu

sdm = pytest.importorskip("sparse_state_linear_gb300")


@pytest.mark.parametrize("cw,dv", [(16, 64), (32, 64), (64, 128)])
def test_row_traffic_moves_whole_pieces_within_chain(cw, dv):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    dev = "cuda:0"
    chains, rows, T, loads, stores = 3, 1000, 5, 20, 12
    # Every element names its own (chain, row, column): exact in fp32 (< 2^24).
    src = torch.arange(chains * rows * dv, dtype=torch.float32, device=dev).view(chains, rows, dv)
    dst = torch.full_like(src, -1.0)
    nbytes = sdm.sdm_measure_row_traffic(src, dst, cw, T, loads, stores, seed=3)
    torch.cuda.synchronize()
    assert sdm.sdm_get_device_status() == 0
    assert nbytes == chains * dv * T * (loads + stores) * 4
    d = dst.cpu().numpy().reshape(chains, rows, dv // cw, cw)
    written = (d != -1.0)
    # A piece is written whole or not at all.
    assert np.all(written.all(axis=-1) == written.any(axis=-1))
    pieces = written.all(axis=-1)
    assert 0 < pieces.sum() <= chains * (dv // cw) * T * stores
    col = np.arange(cw)
    for c, r, sl in zip(*np.nonzero(pieces)):
        p = d[c, r, sl]
        first = int(p[0])
        src_row, rem = divmod(first - c * rows * dv, dv)
        assert rem == sl * cw and 0 <= src_row < rows            # same chain and columns
        assert np.array_equal(p, first + col)                    # unaltered, contiguous
