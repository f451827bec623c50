"""Failure paths without a GPU fault: host-side argument rejection (nothing is
launched), device-side input checks that end the kernel before any access,
and a grid barrier that runs out of time and reports MTP_ERR_TIMEOUT."""
import numpy as np
import pytest

import synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from mtp_speculative_decoding_gb300 import build
    build.build()


def test_barrier_timeout_is_reported_and_context_survives():
    import torch
    import mtp_speculative_decoding_gb300 as mtp
    ws = mtp.alloc_workspace(4096)
    mtp.debug_barrier_timeout(ws, 2000)
    assert mtp.last_error(ws) == mtp.MTP_ERR_TIMEOUT
    x = torch.ones(1024, device="cuda")
    assert float((x * 2).sum()) == 2048.0


def test_host_rejects_bad_arguments():
    import torch
    import mtp_speculative_decoding_gb300 as mtp
    lg = torch.zeros(2, 3, 100, device="cuda")
    dr = torch.zeros(2, 2, dtype=torch.int32, device="cuda")
    out = torch.zeros(2, 3, dtype=torch.int32, device="cuda")
    n = torch.zeros(2, dtype=torch.int32, device="cuda")
    small = mtp.alloc_workspace(64)
    with pytest.raises(mtp.MTPError) as e:
        mtp.verify_greedy(lg, dr, out, n, small)
    assert e.value.code == mtp.MTP_ERR_WORKSPACE
    ws = mtp.alloc_workspace(mtp.workspace_size(None, 2, 2, 100))
    with pytest.raises(mtp.MTPError) as e:
        mtp.verify_sample(lg, lg[:, :2], dr, None, (0.0, 1.0, 0.1, 1.0, 0.0, 0), 0, 0, out, n, ws)
    assert e.value.code == mtp.MTP_ERR_ARG
    with pytest.raises(mtp.MTPError) as e:
        mtp.verify_sample(lg, lg[:, :2], dr, None, (0.7, 1.0, 0.1, 1.0, 0.0, 5), 0, 0, out, n, ws)
    assert e.value.code == mtp.MTP_ERR_UNSUPPORTED


def test_device_rejects_out_of_range_inputs():
    import torch
    import mtp_speculative_decoding_gb300 as mtp
    from mtp_speculative_decoding_gb300.device import upload_draft
    m = synth.ModelSpec(d_t=64, d_a=32, n_blocks=1, n_q_heads=2, head_dim=32, n_kv_heads=1, d_ff=64,
                        vocab=100, dtype="f32", block_view=(0,))
    w = synth.make_draft_workload("bad", m, [synth.ViewSpec(cap=16, window=0, rope_theta=1e4)], 2, 2, [4, 16], 1)
    dev = upload_draft(w)
    drafts = torch.full((2, 2), -7, dtype=torch.int32, device="cuda")
    dev.kv_len[1] = 17        # beyond the full view's capacity
    dev.run(drafts)
    assert mtp.last_error(dev.ws) == mtp.MTP_ERR_ARG
    assert int(drafts.min()) == -7 and int(drafts.max()) == -7
    dev.kv_len[1] = 16
    dev.last_tok[0] = 100     # token id out of range
    dev.run(drafts)
    assert mtp.last_error(dev.ws) == mtp.MTP_ERR_ARG
    dev.last_tok[0] = 3
    dev.run(drafts)
    assert mtp.last_error(dev.ws) == 0 and int(drafts.min()) >= 0
