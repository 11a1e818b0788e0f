"""The five workloads and random layouts, as segment tables plus bf16 tensors.

A layout describes each batch row b as K segments laid end to end along the
sequence axis: segment k spans ``seg_frames[b, k]`` latent frames, of which the
first ``seg_valid[b, k]`` are real and the rest are zero padding.  Each frame
is ``tokens_per_frame`` tokens; positions past the last segment up to ``L``
are padding too.  Zero-padding episodes to a shared frame count is one
segment per row ("lingbot_va_packing" §2.1, make_pad_collate); concatenating
episodes along the sequence axis is several segments in one row
("lingbot_va_attn_profiling", the packing proposal at the end of the page).

Workloads (seed = 1000 + workload number):

1. ``tiny``: B=2, valid frames {5, 3} padded to 8, 32 tokens/frame, L=256,
   H=2, D=64; Q/K/V/dO drawn in fp32 and rounded once to bf16.
2. ``same_length``: B=4 episodes of F=120, 38 tokens/frame, L=4560, H=12,
   D=128, no padding ("lingbot_va_packing" §3.1, same-length batch).
3. ``padded``: B=4 with valid frames {119, 177, 285, 239} padded to 288,
   L=10944, H=12, D=128 ("lingbot_va_packing" §3.1, different-length batch).
4. ``concat64k``: one row of K=7 episodes, F_k = round_up(U{103..362}, 8),
   all frames real, laid end to end and padded to 65,536 tokens; the draw of
   all seven is repeated from the same generator until they fit.
5. ``bucket_sweep``: 40 batches of 4 from the length-bucketing sampler over
   160 lengths F ~ U{103..362}, pool 200, each batch padded to
   round_up(max F, 8).

Cross attention ("lingbot_va_packing" §2.1: the latent and the action tokens
carry their own seq_ids): a ``CrossLayout`` pairs a query layout (the latent
stream) with a key stream over the same segment table at its own tokens per
frame and length.  The pages give no action-token count; 16 per latent frame
is this build's choice.  Cross workloads: workloads 2, 3 and 4 as queries,
keys at 16 tokens per frame, key length the longest row rounded up to 64.

Values are standard normal (numpy PCG64, platform independent) rounded to bf16
with round-to-nearest-even; the upstream gradient dO is drawn on every row,
padding rows included, so a leak through padding would show.
"""

from __future__ import annotations

import dataclasses

import numpy as np
import torch

from .sampler import LengthBucketBatchSampler

TOKENS_PER_FRAME = 38
ACTION_TOKENS_PER_FRAME = 16
PAD_MULTIPLE = 8
F_MIN, F_MAX = 103, 362
SEQ_CAP = 65536


def round_up(x, m):
    return -(-np.asarray(x) // m) * m


@dataclasses.dataclass
class Layout:
    name: str
    seg_frames: np.ndarray  # int32 [B, K]
    seg_valid: np.ndarray   # int32 [B, K]
    tokens_per_frame: int
    L: int
    H: int
    D: int
    seed: int
    fp32_source: bool = False  # draw fp32, round once to bf16 (workload 1)

    @property
    def B(self) -> int:
        return int(self.seg_frames.shape[0])

    @property
    def K(self) -> int:
        return int(self.seg_frames.shape[1])

    def describe(self) -> dict:
        return {
            "name": self.name, "B": self.B, "K": self.K, "L": self.L, "H": self.H,
            "D": self.D, "tokens_per_frame": self.tokens_per_frame,
            "seg_frames": self.seg_frames.tolist(), "seg_valid": self.seg_valid.tolist(),
        }


def _layout(name, frames, valid, T, L, H, D, seed, fp32_source=False) -> Layout:
    frames = np.asarray(frames, dtype=np.int32).reshape(len(frames), -1)
    valid = np.asarray(valid, dtype=np.int32).reshape(frames.shape)
    return Layout(name, frames, valid, int(T), int(L), int(H), int(D), int(seed), fp32_source)


def concat64k_frames(seed: int, k: int = 7, tokens_per_frame: int = TOKENS_PER_FRAME,
                     cap: int = SEQ_CAP) -> np.ndarray:
    rng = np.random.default_rng(seed)
    while True:
        f = round_up(rng.integers(F_MIN, F_MAX + 1, size=k), PAD_MULTIPLE)
        if int(f.sum()) * tokens_per_frame <= cap:
            return f.astype(np.int32)


def config_layout(n: int) -> Layout:
    """Layout of workload ``n`` in 1..4 (workload 5 is ``bucket_sweep_layouts``)."""
    seed = 1000 + n
    T = TOKENS_PER_FRAME
    if n == 1:
        return _layout("tiny", [[8], [8]], [[5], [3]], 32, 256, 2, 64, seed, fp32_source=True)
    if n == 2:
        return _layout("same_length", [[120]] * 4, [[120]] * 4, T, 120 * T, 12, 128, seed)
    if n == 3:
        valid = np.array([119, 177, 285, 239])
        fpad = int(round_up(valid.max(), PAD_MULTIPLE))
        return _layout("padded", [[fpad]] * 4, valid.reshape(4, 1), T, fpad * T, 12, 128, seed)
    if n == 4:
        f = concat64k_frames(seed)
        return _layout("concat64k", f.reshape(1, -1), f.reshape(1, -1), T, SEQ_CAP, 12, 128, seed)
    raise ValueError(f"no single layout for workload {n}")


def bucket_sweep_lengths(seed: int = 1005, n: int = 160) -> np.ndarray:
    return np.random.default_rng(seed).integers(F_MIN, F_MAX + 1, size=n)


def bucket_sweep_layouts(seed: int = 1005, n_episodes: int = 160, batch_size: int = 4,
                         pool: int = 200, H: int = 12, D: int = 128):
    """Workload 5: returns (layouts, batches, lengths), one padded layout per batch."""
    lengths = bucket_sweep_lengths(seed, n_episodes)
    sampler = LengthBucketBatchSampler(lengths, batch_size, 0, 1, seed, pool // batch_size)
    batches = sampler.batches()
    layouts = []
    for i, batch in enumerate(batches):
        f = lengths[batch]
        fpad = int(round_up(f.max(), PAD_MULTIPLE))
        layouts.append(_layout(f"bucket{i:02d}", [[fpad]] * len(batch), f.reshape(-1, 1),
                               TOKENS_PER_FRAME, fpad * TOKENS_PER_FRAME, H, D, seed * 100 + i))
    return layouts, batches, lengths


def random_layout(rng: np.random.Generator, B: int, K: int, T: int, L: int, H: int, D: int,
                  name: str = "random") -> Layout:
    """Random segment table that fits in L: frames >= 0, 0 <= valid <= frames.

    Per row, K sorted cut points in [0, L // T] give the segment frame counts
    (so their sum never exceeds L // T); valid counts are uniform in [0, frames].
    Zero-frame segments, fully padded segments and a padded tail all occur.
    """
    cap = L // T
    frames = np.zeros((B, K), np.int32)
    valid = np.zeros((B, K), np.int32)
    for b in range(B):
        cuts = np.sort(rng.integers(0, cap + 1, size=K))
        frames[b] = np.diff(np.concatenate([[0], cuts]))
        valid[b] = [int(rng.integers(0, f + 1)) for f in frames[b]]
    return _layout(name, frames, valid, T, L, H, D, int(rng.integers(1 << 30)))


def make_tensors(layout: Layout, device="cpu", with_grad_out: bool = True):
    """Q, K, V (and dO) as bf16 [B, L, H, D] tensors drawn from ``layout.seed``."""
    rng = np.random.default_rng(layout.seed)
    shape = (layout.B, layout.L, layout.H, layout.D)
    names = ["q", "k", "v"] + (["do"] if with_grad_out else [])
    out = {}
    for nm in names:
        x = rng.standard_normal(size=shape, dtype=np.float32)
        out[nm] = torch.from_numpy(x).to(torch.bfloat16).to(device)
    return out


@dataclasses.dataclass
class CrossLayout:
    """Queries over ``q`` (its segments, tokens per frame and length); keys and
    values over the same segments at ``tokens_per_frame_k`` tokens per frame
    and length ``Lk``."""
    q: Layout
    tokens_per_frame_k: int
    Lk: int

    @property
    def name(self) -> str:
        return "cross_" + self.q.name

    @property
    def B(self) -> int:
        return self.q.B

    @property
    def H(self) -> int:
        return self.q.H

    @property
    def D(self) -> int:
        return self.q.D

    @property
    def Lq(self) -> int:
        return self.q.L


def cross_layout(q: Layout, tokens_per_frame_k: int = ACTION_TOKENS_PER_FRAME, Lk: int | None = None) -> CrossLayout:
    """Key length: the longest row rounded up to 64 by default; an explicit
    Lk is raised to the longest row if it is shorter."""
    need = int(q.seg_frames.sum(axis=1).max()) * int(tokens_per_frame_k)
    if Lk is None:
        Lk = int(round_up(need, 64))
    return CrossLayout(q, int(tokens_per_frame_k), max(int(Lk), need, 1))


def cross_config_layout(n: int) -> CrossLayout:
    """Cross workload over workload ``n`` in 2..4."""
    if n not in (2, 3, 4):
        raise ValueError(f"no cross layout for workload {n}")
    return cross_layout(config_layout(n))


def make_cross_tensors(cl: CrossLayout, device="cpu", with_grad_out: bool = True):
    """Q (and dO) as bf16 [B, Lq, H, D], K and V as bf16 [B, Lk, H, D], drawn
    in the order q, k, v, dO from the query layout's seed + 7."""
    rng = np.random.default_rng(cl.q.seed + 7)
    out = {}
    for nm in ["q", "k", "v"] + (["do"] if with_grad_out else []):
        L = cl.Lk if nm in ("k", "v") else cl.Lq
        x = rng.standard_normal(size=(cl.B, L, cl.H, cl.D), dtype=np.float32)
        out[nm] = torch.from_numpy(x).to(torch.bfloat16).to(device)
    return out


def make_loss_tensors(B: int, L: int, C: int, seed: int, device="cpu"):
    """Prediction and target of the loss as bf16 [B, L, C] tensors: standard
    normal draws from ``seed`` (prediction first)."""
    rng = np.random.default_rng(seed)
    out = {}
    for nm in ("pred", "target"):
        x = rng.standard_normal(size=(B, L, C), dtype=np.float32)
        out[nm] = torch.from_numpy(x).to(torch.bfloat16).to(device)
    return out

