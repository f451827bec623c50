"""mtp_verify_greedy_noalloc: greedy verify for callers that may not allocate
device memory (its scratch is a small array built into the library instead of
a caller workspace).  Checked through the C ABI against mtp_verify_greedy on
two calls in a row (integer outputs: bit-exact), plus its size limit.  This
file is collected last on purpose."""
import numpy as np
import pytest

import synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from mtp_speculative_decoding_gb300 import build
    build.build()


def _run_both(inp):
    import torch
    import mtp_speculative_decoding_gb300 as mtp
    from mtp_speculative_decoding_gb300.device import to_device
    B, R, V = inp.logits.shape
    lg = to_device(inp.logits, inp.dtype)
    dr = torch.from_numpy(np.ascontiguousarray(inp.drafts, dtype=np.int32)).cuda()
    ref_t = torch.full((B, R), -9, dtype=torch.int32, device="cuda")
    ref_n = torch.full((B,), -9, dtype=torch.int32, device="cuda")
    ws = mtp.alloc_workspace(mtp.workspace_size(None, B, R - 1, V))
    mtp.verify_greedy(lg, dr, ref_t, ref_n, ws)
    got_t = torch.full((B, R), -9, dtype=torch.int32, device="cuda")
    got_n = torch.full((B,), -9, dtype=torch.int32, device="cuda")
    mtp.verify_greedy_noalloc(lg, dr, got_t, got_n)
    torch.cuda.synchronize()
    return ref_t.cpu().numpy(), ref_n.cpu().numpy(), got_t.cpu().numpy(), got_n.cpu().numpy()


def test_noalloc_matches_workspace_verify_on_two_calls_in_a_row():
    # the second call reuses the scratch the first left behind: it must clear it
    first = synth.make_verify_greedy_inputs(1)                                  # B 1, N 3, V 262144 bf16
    second = synth.make_verify_greedy_inputs(0, seed=77, B=40, N=4, V=5003, dtype="f32")
    for inp in (first, second):
        rt, rn, gt, gn = _run_both(inp)
        assert np.array_equal(gt, rt) and np.array_equal(gn, rn)
        assert np.array_equal(gn, inp.planted)


def test_noalloc_rejects_sizes_beyond_its_scratch():
    import torch
    import mtp_speculative_decoding_gb300 as mtp
    B, N, V = 64, 8, 100            # 64 * 9 = 576 rows > 480
    lg = torch.zeros((B, N + 1, V), dtype=torch.float32, device="cuda")
    dr = torch.zeros((B, N), dtype=torch.int32, device="cuda")
    out = torch.full((B, N + 1), -9, dtype=torch.int32, device="cuda")
    n = torch.full((B,), -9, dtype=torch.int32, device="cuda")
    with pytest.raises(mtp.MTPError) as e:
        mtp.verify_greedy_noalloc(lg, dr, out, n)
    assert e.value.code == mtp.MTP_ERR_UNSUPPORTED
    assert int(out.min()) == -9 and int(n.min()) == -9
