"""The measurement kernels the bench's rooflines are taken against run to
completion, touch only what they promise, and report what they move.

* nsa_probe_l2_gather: random-block copies; every CTA records its SM and a
  start no later than its end; bytes = ctas x warps x loads x tile bytes.
* nsa_probe_gather_rows: the forward's copies for an index tensor, for
  every depth the bench sweeps, with and without unused shared memory.
* nsa_probe_reduce_rows: adds zeros, so the buffer is unchanged.
"""

import numpy as np
import pytest

from _parity import small_inputs, to_dev

pytestmark = pytest.mark.gpu


def test_random_block_probe_records_and_bytes():
    import torch

    from nsa_block_selection_gb300 import _lib

    k = torch.randn((4096, 8, 128), device="cuda").half()
    v = torch.randn_like(k)
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    for rows in (16, 32, 64):
        rec = torch.full((sms, 3), -1, dtype=torch.int64, device="cuda")
        n = _lib.probe_l2_gather(k, v, 0, 64, sms, 4, 2, 40, record=rec, rows_per_box=rows)
        torch.cuda.synchronize()
        assert _lib.sync_status() == 0
        assert n == sms * 4 * 40 * 2 * rows * 128
        r = rec.cpu().numpy()
        assert (r[:, 0] >= 0).all() and (r[:, 0] < sms).all()
        assert (r[:, 1] > 0).all() and (r[:, 2] >= r[:, 1]).all()
    # all groups interleaved (g = -1), 32-key blocks
    _lib.probe_l2_gather(k, v, -1, 32, sms, 8, 1, 40)
    torch.cuda.synchronize()
    assert _lib.sync_status() == 0


@pytest.mark.parametrize("cfg", [(4, 4, 2), (32, 1, 1), (16, 1, 2), (2, 4, 6)])
def test_rows_probe_runs_on_padded_and_ragged_rows(cfg):
    import torch

    from nsa_block_selection_gb300 import _lib

    q, k, v, idx = small_inputs(2, 777, 700, 16, 2, 128, 64, 6, "first_two_local", seed=3)
    idx = idx.copy()
    idx[0, 5:9] = -1                       # empty rows
    idx[1, 10, 1, 0] = 1 << 20             # an out-of-range id: padding
    tk, tv, ti = to_dev(k, v, idx)
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    warps, cps, slots = cfg
    for pad in (0, 4096):
        _lib.probe_gather_rows(tk, tv, ti, 64, sms * cps, warps, slots, extra_smem_bytes=pad)
        torch.cuda.synchronize()
        assert _lib.sync_status() == 0


def test_reduce_probe_adds_zeros():
    import torch

    from nsa_block_selection_gb300 import _lib

    rows, stride = 2048, 4096
    buf = torch.randn(rows * stride, device="cuda")
    before = buf.clone()
    n = _lib.probe_reduce_rows(buf, rows, stride, 64, 4, 8)
    torch.cuda.synchronize()
    assert n == 64 * 4 * 8 * 4096
    assert torch.equal(buf, before)
    assert np.isfinite(buf.cpu().numpy()).all()
