"""Greedy draft-block verification on the GPU: (accept_len, next_token) must
equal the oracle's bit for bit on identical logits.

Rule (SpecPilot summary, airadar.tv English edition, "Risks" bullet 3: every
committed token is the target's greedy choice): per position the lowest index
of the row maximum; accept the longest agreeing draft prefix; the next token
is the target's token at the first disagreement.
"""
import numpy as np
import pytest

from helpers import check_gemm, to_dev_bits
from lossless_bit_weight_w12_gb300 import synth

pytestmark = pytest.mark.gpu


def _verify(w12mod, dev, lg, R, T, draft):
    import torch
    V = lg.shape[1]
    if lg.dtype == np.uint16:
        lg_d = to_dev_bits(lg, dev).view(torch.bfloat16)
    else:
        lg_d = torch.from_numpy(np.ascontiguousarray(lg)).to(dev)
    dr_d = torch.from_numpy(np.ascontiguousarray(draft, dtype=np.int32)).to(dev)
    acc = torch.full((R,), -7, dtype=torch.int32, device=dev)
    nxt = torch.full((R,), -7, dtype=torch.int32, device=dev)
    ws = w12mod.workspace(w12mod.verify_workspace_size(R, T, V), dev)
    w12mod.verify_greedy(lg_d, R, T, dr_d if T > 1 else None, acc, nxt, ws)
    return acc.cpu().numpy(), nxt.cpu().numpy()


@pytest.mark.parametrize("dtype", [np.float32, np.uint16], ids=["f32", "bf16"])
@pytest.mark.parametrize("R,T,V", [(1, 16, 151936), (2, 16, 32000), (8, 16, 4099),
                                   (1, 1, 1000), (3, 2, 7), (1, 16, 1), (16, 8, 151936)])
def test_verify_vs_oracle(dev, w12mod, oracle, dtype, R, T, V):
    rng = synth.streams(500 + R * 7 + T + V % 97, 2)
    lg = synth.logits(rng[0], R * T, V, dtype=dtype)
    g = oracle.argmax(lg).reshape(R, T)
    draft = synth.draft_tokens(rng[1], g, R, T, V)
    want = oracle.verify_greedy(lg, R, T, draft)
    got = _verify(w12mod, dev, lg, R, T, draft)
    np.testing.assert_array_equal(got[0], want[0])
    np.testing.assert_array_equal(got[1], want[1])


def test_verify_ties_nan_signed_zero(dev, w12mod, oracle):
    R, T, V = 4, 5, 3000
    lg = np.full((R * T, V), -1.0, dtype=np.float32)
    lg[0, [17, 2000, 2999]] = 3.5            # three-way tie: lowest index 17
    lg[1, [5, 6]] = [np.inf, np.nan]         # NaN above +Inf
    lg[2, [9, 10]] = [-0.0, 0.0]             # row 2: all -1 except +-0 ... equal
    lg[2, :9] = -5.0
    lg[3, :] = 7.0                           # all equal: index 0
    lg[4, [100, 50]] = [np.nan, np.nan]      # first NaN wins: 50
    lg[5:, :] = np.random.default_rng(0).standard_normal((R * T - 5, V)).astype(np.float32)
    g = oracle.argmax(lg)
    assert g[0] == 17 and g[1] == 6 and g[2] == 9 and g[3] == 0 and g[4] == 50
    gd = g.reshape(R, T)
    drafts = [gd[0, :4], np.r_[gd[1, :2], (gd[1, 2:4] + 1) % V], np.r_[(gd[2, :1] + 1) % V, gd[2, 1:4]],
              (gd[3, :4] + 1) % V]
    draft = np.stack(drafts).astype(np.int32)
    want = oracle.verify_greedy(lg, R, T, draft)
    got = _verify(w12mod, dev, lg, R, T, draft)
    np.testing.assert_array_equal(got[0], want[0])
    np.testing.assert_array_equal(got[1], want[1])
    assert want[0].tolist() == [4, 2, 0, 0]


def test_verify_repeated_calls_reuse_workspace(dev, w12mod, oracle):
    import torch
    R, T, V = 2, 16, 50000
    ws = w12mod.workspace(w12mod.verify_workspace_size(R, T, V), dev)
    for s in range(3):
        rng = synth.streams(900 + s, 2)
        lg = synth.logits(rng[0], R * T, V)
        draft = synth.draft_tokens(rng[1], oracle.argmax(lg).reshape(R, T), R, T, V)
        lg_d = torch.from_numpy(lg).to(dev)
        dr_d = torch.from_numpy(draft).to(dev)
        acc = torch.empty(R, dtype=torch.int32, device=dev)
        nxt = torch.empty(R, dtype=torch.int32, device=dev)
        w12mod.verify_greedy(lg_d, R, T, dr_d, acc, nxt, ws)
        want = oracle.verify_greedy(lg, R, T, draft)
        assert acc.cpu().numpy().tolist() == want[0].tolist()
        assert nxt.cpu().numpy().tolist() == want[1].tolist()


@pytest.mark.parametrize("R,T,K,N", [(1, 16, 256, 5000), (2, 16, 1024, 3001), (1, 1, 128, 77),
                                     (1, 8, 512, 3001), (2, 4, 384, 2000),
                                     (8, 16, 512, 2048), (4, 16, 384, 3000), (3, 13, 256, 2500)])
def test_verify_lmhead_fused(dev, w12mod, oracle, R, T, K, N):
    """Fused lm_head + verify.  Drafts follow the oracle's fp64-logit argmax for
    a geometric prefix; the fused (accept, next) must equal the oracle's verify
    on the kernel's own fp32 logits (returned through logits_out), and those
    logits must match the fp64 product within the GEMM tolerance."""
    import torch
    M = R * T
    rng = synth.streams(700 + K + N + M, 3)
    w = synth.weights(rng[0], K, N)
    hidden = synth.activations(rng[1], M, K)
    od, oblob = oracle.encode(w, oracle.LAYOUT_NK)
    y_ref, s_ref = oracle.gemm(od, oblob, hidden)
    g64 = np.argmax(y_ref, axis=1).reshape(R, T)
    draft = synth.draft_tokens(rng[2], g64, R, T, N)
    d, blob = w12mod.encode(w, w12mod.LAYOUT_NK)
    blob_d = w12mod.upload(blob, dev)
    h_d = to_dev_bits(hidden, dev)
    dr_d = torch.from_numpy(draft).to(dev) if T > 1 else None
    acc = torch.empty(R, dtype=torch.int32, device=dev)
    nxt = torch.empty(R, dtype=torch.int32, device=dev)
    logits = torch.empty((M, N), dtype=torch.float32, device=dev)
    ws = w12mod.workspace(w12mod.verify_lmhead_workspace_size(d, R, T), dev)
    for rep in range(2):  # the second call reuses the workspace
        w12mod.verify_greedy_lmhead(h_d, d, blob_d, R, T, dr_d, acc, nxt, ws, logits_out_dev=logits)
        lg = logits.cpu().numpy()
        check_gemm(lg.astype(np.float64), y_ref, s_ref, what="lm_head logits")
        want = oracle.verify_greedy(lg, R, T, draft)
        assert acc.cpu().numpy().tolist() == want[0].tolist()
        assert nxt.cpu().numpy().tolist() == want[1].tolist()
    # without logits_out the result is the same
    acc2 = torch.empty(R, dtype=torch.int32, device=dev)
    nxt2 = torch.empty(R, dtype=torch.int32, device=dev)
    w12mod.verify_greedy_lmhead(h_d, d, blob_d, R, T, dr_d, acc2, nxt2, ws)
    assert torch.equal(acc, acc2) and torch.equal(nxt, nxt2)
