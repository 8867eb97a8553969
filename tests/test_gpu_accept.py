"""GPU parity of the verify-acceptance entry point (moe_mxfp4_accept) against the oracle.

Targets, accepted lengths and next tokens are integers decided by comparisons of the
same fp32 logits on both sides: they must match bit for bit.
"""
import numpy as np
import pytest
import torch

import mxfp4_moe_expert_gb300 as pkg
from oracle import moe_oracle as O

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    import os
    if not os.path.exists(pkg.LIB_PATH):
        from mxfp4_moe_expert_gb300 import build
        build.build()
    pkg.load_library()


@pytest.mark.parametrize("S,B,V", [(1, 8, 5), (32, 8, 4099), (5, 1, 17), (64, 8, 151936)])
def test_accept_matches_oracle(S, B, V):
    g = torch.Generator().manual_seed(S * 1000 + B * 10 + V)
    lg = torch.randn((S, B, V), generator=g, dtype=torch.float32)
    lg[0, 0, :3] = 5.0                       # ties at the maximum
    if V > 7:
        lg[-1, -1, 7] = float("nan")
    tgt = O.accept_block(lg.double().numpy(), np.zeros((S, B), dtype=np.int64))["target"]
    # drafts that agree with the target for a random prefix of each stream, then differ
    tokens = np.zeros((S, B), dtype=np.int32)
    lens = torch.randint(0, B, (S,), generator=g).numpy()
    for s in range(S):
        tokens[s, 0] = 3
        for i in range(1, B):
            tokens[s, i] = tgt[s, i - 1] if i <= lens[s] else (tgt[s, i - 1] + 1) % V
    ref = O.accept_block(lg.numpy().astype(np.float64), tokens)
    target, acc, nxt = pkg.accept(lg.cuda(), torch.from_numpy(tokens).cuda())
    torch.cuda.synchronize()
    assert np.array_equal(target.cpu().numpy(), ref["target"])
    assert np.array_equal(acc.cpu().numpy(), ref["accepted"])
    assert np.array_equal(nxt.cpu().numpy(), ref["next_token"])
    assert np.array_equal(ref["accepted"], np.minimum(lens, B - 1) + 1)


def test_accept_rejects_bad_sizes():
    lg = torch.zeros((1, 2, 3), device="cuda")
    tok = torch.zeros((1, 2), dtype=torch.int32, device="cuda")
    out = torch.zeros((4,), dtype=torch.int32, device="cuda")
    st = torch.cuda.current_stream().cuda_stream
    assert pkg.moe_mxfp4_accept(lg.data_ptr(), tok.data_ptr(), 1, 0, 3, out.data_ptr(), out.data_ptr(), None,
                                st) == pkg.MOE_ERR_INVALID_ARG
    assert pkg.moe_mxfp4_accept(lg.data_ptr(), tok.data_ptr(), 0, 2, 3, out.data_ptr(), out.data_ptr(), None,
                                st) == pkg.MOE_OK
