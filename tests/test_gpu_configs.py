"""The workloads as stated, end to end on the GPU.

Config 0: one K = N = 1024 linear, M = 1, seed 0 -- encode -> decode
round trip bit-exact, then y = x W in fp32 against the oracle (every output).

Config 4: the full stack -- 64 layers of the 27B-class linears plus the
lm_head 5120 -> 151936 at M = 16 (one draft block of T = 16), seed 4.
 - every layer's six matrices: GPU decode bit-exact against the generated
   weights, and the batched W12 GEMM at M = 16 within the tolerance on
   sampled columns (the oracle encodes and multiplies those columns); at
   layers 0, 31 and 63 every output of all six matrices against the float64
   definition y = x W (numpy on the uncompressed weights);
 - the lm_head: fused greedy verify.  The fp64 reference logits are the
   definition y = h W computed with numpy's float64 matmul on the generated
   (uncompressed) weights; the drafts follow their argmax for a geometric
   prefix (p = 0.7); the kernel's (accept_len, next) must equal the oracle's
   verify on the kernel's own fp32 logits, bit for bit, and those logits must
   be within the GEMM tolerance of the fp64 ones.
Tensor streams: SeedSequence(4).spawn(64 * 6 + 4): layer l, linear i -> 6l + i;
lm_head -> 384; per-layer activations -> 385 (one stream, drawn in order);
hidden -> 386; drafts -> 387.
"""
import numpy as np
import pytest

from helpers import check_gemm, dev_bits_to_np, ref_gemm_f64, to_dev_bits
from lossless_bit_weight_w12_gb300 import synth

pytestmark = pytest.mark.gpu


def test_config0_roundtrip_and_gemm(dev, w12mod, oracle):
    import torch
    rng = synth.streams(0, 2)
    w = synth.weights(rng[0], 1024, 1024)
    x = synth.activations(rng[1], 1, 1024)
    d, blob = w12mod.encode(w, w12mod.LAYOUT_NK)
    od, oblob = oracle.encode(w, oracle.LAYOUT_NK)
    assert blob.tobytes() == oblob.tobytes()
    blob_d = w12mod.upload(blob, dev)
    out = torch.empty((1024, 1024), dtype=torch.int16, device=dev)
    w12mod.decode(d, blob_d, out, w12mod.LAYOUT_NK)
    np.testing.assert_array_equal(dev_bits_to_np(out), w)
    y = torch.empty((1, 1024), dtype=torch.float32, device=dev)
    ws = w12mod.workspace(w12mod.gemm_workspace_size(d, 1), dev)
    w12mod.gemm(d, blob_d, to_dev_bits(x, dev), y, ws)
    y_ref, s_ref = oracle.gemm(od, oblob, x)
    check_gemm(y.cpu().numpy().astype(np.float64), y_ref, s_ref, what="config 0")


def _bf16_f64(u):
    return (np.asarray(u, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def test_config4_full_stack(dev, w12mod, oracle):
    import torch
    L, M = synth.N_LAYERS_STACK, 16
    shapes = synth.LAYER_SHAPES
    rngs = synth.streams(4, 6 * L + 4)
    x_rng = rngs[6 * L + 1]
    descs_ws = None
    for layer in range(L):
        descs, blobs, xs, ws_np = [], [], [], []
        for i, (name, K, N) in enumerate(shapes):
            w = synth.weights(rngs[6 * layer + i], K, N)
            d, blob = w12mod.encode(w, w12mod.LAYOUT_NK)
            b = w12mod.upload(blob, dev)
            out = torch.empty((N, K), dtype=torch.int16, device=dev)
            w12mod.decode(d, b, out, w12mod.LAYOUT_NK)
            ref = torch.from_numpy(w.view(np.int16)).to(dev)
            assert torch.equal(out, ref), f"layer {layer} {name}: decode differs"
            del out, ref
            descs.append(d)
            blobs.append(b)
            xs.append(synth.activations(x_rng, M, K))
            ws_np.append(w)
        ys = [torch.empty((M, N), dtype=torch.float32, device=dev) for _, _, N in shapes]
        if descs_ws is None:
            descs_ws = w12mod.workspace(w12mod.gemm_batched_workspace_size(descs, M), dev)
        w12mod.gemm_batched(descs, blobs, [to_dev_bits(x, dev) for x in xs], ys, descs_ws)
        torch.cuda.synchronize()
        assert w12mod.get_device_error(descs_ws) == 0
        pick = np.random.default_rng(layer)
        for i, (name, K, N) in enumerate(shapes):
            y = ys[i].cpu().numpy().astype(np.float64)
            assert np.isfinite(y).all(), f"layer {layer} {name}"
            if layer in (0, L - 1) or i == layer % 6:  # oracle on sampled columns
                ns = np.unique(np.r_[pick.integers(0, N, 6), [N - 1]])
                y_ref, s_ref = oracle.gemm(*oracle.encode(ws_np[i][ns], oracle.LAYOUT_NK), xs[i])
                check_gemm(y[:, ns], y_ref, s_ref, what=f"config 4 layer {layer} {name}")
            if layer in (0, L // 2 - 1, L - 1):  # every output against the float64 definition
                (y_ref, s_ref), = ref_gemm_f64(ws_np[i], [xs[i]])
                check_gemm(y, y_ref, s_ref, what=f"config 4 layer {layer} {name} (every output)")
        del blobs, ys, ws_np

    # lm_head + fused greedy verify
    K, N = synth.LM_HEAD_SHAPE[1], synth.LM_HEAD_SHAPE[2]
    R, T = 1, 16
    w = synth.weights(rngs[6 * L], K, N)
    hidden = synth.activations(rngs[6 * L + 2], R * T, K)
    hf = _bf16_f64(hidden)
    y64 = np.empty((R * T, N), dtype=np.float64)
    s64 = np.empty((R * T, N), dtype=np.float64)
    for c0 in range(0, N, 8192):
        wf = _bf16_f64(w[c0:c0 + 8192])            # [cols, K]
        y64[:, c0:c0 + 8192] = hf @ wf.T
        s64[:, c0:c0 + 8192] = np.abs(hf) @ np.abs(wf).T
    g64 = np.argmax(y64, axis=1).reshape(R, T)
    draft = synth.draft_tokens(rngs[6 * L + 3], g64, R, T, N)
    d, blob = w12mod.encode(w, w12mod.LAYOUT_NK)
    b = w12mod.upload(blob, dev)
    acc = torch.empty(R, dtype=torch.int32, device=dev)
    nxt = torch.empty(R, dtype=torch.int32, device=dev)
    logits = torch.empty((R * T, N), dtype=torch.float32, device=dev)
    ws = w12mod.workspace(w12mod.verify_lmhead_workspace_size(d, R, T), dev)
    w12mod.verify_greedy_lmhead(to_dev_bits(hidden, dev), d, b, R, T,
                                torch.from_numpy(draft).to(dev), acc, nxt, ws, logits_out_dev=logits)
    lg = logits.cpu().numpy()
    check_gemm(lg.astype(np.float64), y64, s64, what="config 4 lm_head logits")
    want = oracle.verify_greedy(lg, R, T, draft)
    assert acc.cpu().numpy().tolist() == want[0].tolist()
    assert nxt.cpu().numpy().tolist() == want[1].tolist()
    # positions whose fp32-logit argmax differs from the fp64 one (near-ties only)
    flips = int((oracle.argmax(lg) != g64.reshape(-1)).sum())
    assert flips <= 2, f"{flips} argmax flips between fp32 and fp64 logits"
