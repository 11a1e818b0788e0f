"""masked_mse_loss / masked_mse_loss_bwd (the frame_valid-masked loss,
"lingbot_va_packing" §2.1 compute_loss) against the fp64 oracle (GPU).

The mask reaches the oracle from the page's rule (frame_valid = f <
valid_frames[b]) on pad-collated rows and from the oracle's own seq_ids on
concatenated rows; the kernels take the seq_ids the library builds.

Tolerances, from the arithmetic: the loss is a sum of fp32 squares of exact
bf16 differences, added in fp32 inside a warp and as pairs of fp32 values
(about 48 significant bits) across warps and CTAs, so its relative error is
~1e-6; the test allows 1e-5.  The gradient is rounded once to bf16 (2^-9
relative): per element |err| <= 2^-8 |ref| + 1e-30, exact zeros on padding
tokens.
"""

import numpy as np
import pytest
import torch

import oracle
import workloads as wl

pytestmark = pytest.mark.gpu

LOSS_REL = 1e-5


@pytest.fixture(scope="module")
def pvl(cuda_ok):
    import packed_variable_length_gb300 as p
    return p


def to_np(t):
    return t.detach().to("cpu", torch.float64).numpy()


def check_grad(got, ref, valid):
    assert np.isfinite(got).all()
    assert not got[~valid].any(), "gradient on padding tokens"
    err = np.abs(got - ref)
    bad = err > 2.0 ** -8 * np.abs(ref) + 1e-30
    assert not bad.any(), f"{bad.sum()} gradient elements out of tolerance, worst {err.max():.3e}"


def run_case(pvl, seg_frames, seg_valid, T, L, C, seed, mask_ref=None, grad_scale=1.0):
    seg_frames = np.asarray(seg_frames)
    seg_valid = np.asarray(seg_valid)
    B = seg_frames.shape[0]
    t = wl.make_loss_tensors(B, L, C, seed)
    sid = pvl.pack_build_seq_ids(seg_frames, seg_valid, T, L)
    pred, target = t["pred"].cuda(), t["target"].cuda()
    loss, grad = pvl.masked_mse_loss(pred, target, sid, grad=True, grad_scale=grad_scale)
    pvl.device_error()
    valid = mask_ref if mask_ref is not None else oracle.valid_from_seq_id(
        oracle.build_seq_ids(seg_frames, seg_valid, T, L))
    ref, n = oracle.masked_mse(t["pred"], t["target"], valid)
    got = float(loss.item())
    if n == 0:
        assert got == 0.0
    else:
        assert abs(got - ref) <= LOSS_REL * abs(ref), (got, ref)
    check_grad(to_np(grad), oracle.masked_mse_grad(t["pred"], t["target"], valid, dloss=grad_scale), valid)
    return pred, target, sid, loss, grad, valid


@pytest.mark.parametrize("n", [2, 3])
@pytest.mark.parametrize("C", [8, 48, 192])
def test_pad_collated_workloads(pvl, n, C):
    """Workloads 2 and 3 (B = 4 episodes padded to a shared F): the oracle's
    mask is the page's frame_valid rule spread over the frame's tokens."""
    lay = wl.config_layout(n)
    F = int(lay.seg_frames[0, 0])
    T = 8 if C == 192 else lay.tokens_per_frame   # keep the case small
    valid = oracle.frame_valid_tokens(lay.seg_valid[:, 0], F, T)
    run_case(pvl, lay.seg_frames, lay.seg_valid, T, F * T, C, seed=4000 + n, mask_ref=valid)


def test_concat64k_latent_grid(pvl):
    """The measured case: the 64k pack's seven episodes on the latent grid
    (8 x 16 positions per frame, C = 48), tail padding to the pack's frame
    capacity."""
    lay = wl.config_layout(4)
    frames = lay.L // lay.tokens_per_frame
    pred, target, sid, loss, grad, _ = run_case(pvl, lay.seg_frames, lay.seg_valid, 128, frames * 128, 48,
                                                seed=4004)
    # the loss alone (no grid barrier: the last CTA reads the count) and the
    # gradient alone give the same bits as the fused call, over a full grid
    loss_only = pvl.masked_mse_loss(pred, target, sid)
    grad_only = pvl.masked_mse_loss_bwd(pred, target, sid, torch.ones(1, device="cuda"))
    pvl.device_error()
    assert torch.equal(loss_only, loss)
    assert torch.equal(grad_only, grad)


def test_random_layouts(pvl):
    rng = np.random.default_rng(4100)
    for i in range(8):
        B, K = int(rng.integers(1, 5)), int(rng.integers(1, 5))
        T = int(rng.integers(1, 40))
        C = int(rng.choice([8, 16, 24, 48, 520]))
        frames = rng.integers(0, 12, size=(B, K))
        valid = np.minimum(frames, rng.integers(0, 12, size=(B, K)))
        L = max(1, int(frames.sum(axis=1).max()) * T + int(rng.integers(0, 50)))
        run_case(pvl, frames, valid, T, L, C, seed=4100 + i, grad_scale=float(rng.uniform(-2, 2)))


def test_degenerate(pvl):
    # no valid token: loss 0, gradient 0
    run_case(pvl, [[4, 4]], [[0, 0]], 3, 30, 8, seed=1)
    # one valid token of one row
    run_case(pvl, [[1], [2]], [[1], [0]], 1, 5, 16, seed=2)
    # a single token, a single vector
    run_case(pvl, [[1]], [[1]], 1, 1, 8, seed=3)
    # every token valid, odd token count (ids not a multiple of 4)
    run_case(pvl, [[7]], [[7]], 3, 21, 8, seed=4)


def test_padding_is_never_read(pvl):
    """NaN in pred and target on padding tokens changes nothing: the kernel
    does not read them."""
    lay = wl.config_layout(3)
    F = int(lay.seg_frames[0, 0])
    T, C = 4, 16
    L = F * T
    sid = pvl.pack_build_seq_ids(lay.seg_frames, lay.seg_valid, T, L)
    t = wl.make_loss_tensors(lay.B, L, C, 77)
    pred, target = t["pred"].cuda(), t["target"].cuda()
    loss0, grad0 = pvl.masked_mse_loss(pred, target, sid, grad=True)
    pad = (sid < 0)
    pred[pad] = float("nan")
    target[pad] = float("nan")
    loss1, grad1 = pvl.masked_mse_loss(pred, target, sid, grad=True)
    pvl.device_error()
    assert torch.equal(loss0, loss1)
    assert torch.equal(grad0, grad1)


def test_fused_and_separate_gradient_agree(pvl):
    """grad_scale on the host and dloss on the device give the same bits;
    the loss is deterministic run to run."""
    lay = wl.config_layout(2)
    F = int(lay.seg_frames[0, 0])
    T, C = 38, 48
    sid = pvl.pack_build_seq_ids(lay.seg_frames, lay.seg_valid, T, F * T)
    t = wl.make_loss_tensors(lay.B, F * T, C, 5)
    pred, target = t["pred"].cuda(), t["target"].cuda()
    loss_a, grad_a = pvl.masked_mse_loss(pred, target, sid, grad=True, grad_scale=0.37)
    grad_b = pvl.masked_mse_loss_bwd(pred, target, sid, torch.tensor([0.37], device="cuda"))
    loss_c = pvl.masked_mse_loss(pred, target, sid)
    pvl.device_error()
    assert torch.equal(grad_a, grad_b)
    assert torch.equal(loss_a, loss_c)


def test_autograd(pvl):
    lay = wl.config_layout(3)
    F = int(lay.seg_frames[0, 0])
    T, C = 2, 24
    L = F * T
    sid = pvl.pack_build_seq_ids(lay.seg_frames, lay.seg_valid, T, L)
    t = wl.make_loss_tensors(lay.B, L, C, 9)
    pred = t["pred"].cuda().requires_grad_(True)
    target = t["target"].cuda()
    loss = pvl.frame_valid_mse(pred, target, sid)
    (0.3 * loss).backward()
    pvl.device_error()
    valid = oracle.frame_valid_tokens(lay.seg_valid[:, 0], F, T)
    ref, _ = oracle.masked_mse(t["pred"], t["target"], valid)
    assert loss.dim() == 0 and abs(loss.item() - ref) <= LOSS_REL * ref
    check_grad(to_np(pred.grad), oracle.masked_mse_grad(t["pred"], t["target"], valid, dloss=0.3), valid)
