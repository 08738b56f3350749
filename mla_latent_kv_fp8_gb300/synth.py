"""Seeded synthetic inputs for paged FP8 latent-KV MLA decode.

This module holds input generation only (random draws, quantisation of the
synthetic latents to FP8 bytes with a library cast, and page placement).  It
contains none of the attention arithmetic, and both the CUDA path's tests and
the FP64 oracle consume the exact bytes it produces.

Recipe (the post's own traces are not available; these shapes stand in):
  * q ~ N(0, 1) in fp32, rounded to bf16 (round-to-nearest-even);
  * latents ~ N(0, 1) in fp32; one per-tensor scale = amax / 448 over every
    generated position; codes = clamp(latent / scale, +-448) cast to
    float8_e4m3fn (RNE) and stored as raw bytes, 576 bytes per position;
  * pages of 64 positions; physical page ids are a random permutation of the
    pool, assigned to requests in order; unused block-table slots hold 0;
  * sm_scale = 1 / sqrt(192).
CPU draws use numpy's PCG64 (identical on x86-64 and aarch64); large caches
are drawn on the GPU with torch's Philox generator when a CUDA device is given.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np
import torch

PAGE = 64
D_QK = 576
D_V = 512
FP8_MAX = 448.0
SM_SCALE = 1.0 / math.sqrt(192.0)
_CHUNK = 8192  # positions per generation chunk (CPU)
_CHUNK_CUDA = 65536  # positions per generation chunk (GPU)


@dataclass
class DecodeCase:
    """One decode call's inputs.  ``seq_lens`` counts the T new positions."""
    q: torch.Tensor            # bf16 [B, T, H, 576]
    kv_cache: torch.Tensor     # uint8 (e4m3fn codes) [num_pages, 64, 576]
    kv_scale: torch.Tensor     # float32 [1]
    block_table: torch.Tensor  # int32 [B, max_pages]
    seq_lens: torch.Tensor     # int32 [B]
    sm_scale: float = SM_SCALE
    lens: list = field(default_factory=list)  # host copy of seq_lens

    @property
    def B(self):
        return self.q.shape[0]

    @property
    def T(self):
        return self.q.shape[1]

    @property
    def H(self):
        return self.q.shape[2]

    def kv_bytes(self) -> int:
        """Latent bytes one decode call must read: 576 per visible position."""
        return kv_bytes_for_lengths(self.lens)

    def to(self, device) -> "DecodeCase":
        return DecodeCase(self.q.to(device), self.kv_cache.to(device), self.kv_scale.to(device),
                          self.block_table.to(device), self.seq_lens.to(device), self.sm_scale,
                          list(self.lens))


def kv_bytes_for_lengths(lens) -> int:
    """576 FP8 bytes per cached position (one byte per latent element, no per-position scale)."""
    return int(sum(int(x) for x in lens)) * D_QK


def mla_payload_bytes(layers: int, positions: int, shards: int = 1) -> float:
    """Latent bytes per GPU for a conversation: layers x positions x 576 / shards."""
    return layers * positions * D_QK / shards


def _normal_chunk(seed_words, n, device):
    """n standard normals (fp32) from a counter-free, seed-addressed stream."""
    if device.type == "cuda":
        g = torch.Generator(device=device)
        s = 0
        for w in seed_words:
            s = (s * 1000003 + int(w) + 1) % (2**63 - 1)
        g.manual_seed(s)
        return torch.randn(n, generator=g, device=device, dtype=torch.float32)
    rng = np.random.default_rng([int(w) for w in seed_words])
    return torch.from_numpy(rng.standard_normal(n, dtype=np.float32))


def _latent_chunk(seed, b, c0, m, device, pattern):
    """Latents of positions c0 .. c0+m-1 of request b, fp32 [m, 576]: N(0,1)
    draws, reshaped by the stress pattern if one is given."""
    x = _normal_chunk((seed, 7, b, c0), m * D_QK, device).view(m, D_QK)
    if pattern is not None:
        x = pattern.latents(b, c0, x)
    return x


def _latent_codes(seed, lens_padded, device, scale=None, pattern=None):
    """Per-request FP8 code blocks [Lpad_b, 576] for N(0,1) latents (or the
    latents of a stress pattern).

    Two passes over the same seed-addressed chunks: amax first (unless a scale
    is supplied), then quantisation.  Returns (list of uint8 tensors, scale)."""
    chunk = _CHUNK_CUDA if device.type == "cuda" else _CHUNK
    if scale is None:
        amax = 0.0
        for b, L in enumerate(lens_padded):
            for c0 in range(0, L, chunk):
                x = _latent_chunk(seed, b, c0, min(chunk, L - c0), device, pattern)
                amax = max(amax, float(x.abs().max()))
        scale = np.float32(amax) / np.float32(FP8_MAX)
    scale = np.float32(scale)
    blocks = []
    st = torch.tensor(float(scale), dtype=torch.float32, device=device)
    for b, L in enumerate(lens_padded):
        out = torch.empty((L, D_QK), dtype=torch.uint8, device=device)
        for c0 in range(0, L, chunk):
            m = min(chunk, L - c0)
            x = _latent_chunk(seed, b, c0, m, device, pattern).reshape(-1)
            y = torch.clamp(x / st, -FP8_MAX, FP8_MAX).to(torch.float8_e4m3fn)
            out[c0:c0 + m] = y.view(torch.uint8).view(m, D_QK)
        blocks.append(out)
    return blocks, float(scale)


def paginate(blocks, seed, device, *, permute=True, max_pages=None, extra_pages=0):
    """Place per-request code blocks ([pages_b*64, 576] uint8) into a page pool.

    Returns (kv_cache [num_pages,64,576], block_table int32 [B,max_pages])."""
    pages = [blk.shape[0] // PAGE for blk in blocks]
    total = sum(pages) + extra_pages
    mp = max(pages) if pages else 0
    if max_pages is None:
        max_pages = max(mp, 1)
    assert max_pages >= mp
    rng = np.random.default_rng([int(seed), 11])
    perm = rng.permutation(total) if permute else np.arange(total)
    kv = torch.zeros((max(total, 1), PAGE, D_QK), dtype=torch.uint8, device=device)
    bt = np.zeros((len(blocks), max_pages), dtype=np.int32)
    off = 0
    for b, blk in enumerate(blocks):
        ids = perm[off:off + pages[b]]
        bt[b, :pages[b]] = ids
        if pages[b]:
            idx = torch.from_numpy(ids.astype(np.int64)).to(device)
            kv[idx] = blk.view(pages[b], PAGE, D_QK)
        off += pages[b]
    return kv, torch.from_numpy(bt).to(device)


def make_q(seed, B, T, H, device="cpu", pattern=None):
    rng = np.random.default_rng([int(seed), 3])
    q = torch.from_numpy(rng.standard_normal((B, T, H, D_QK), dtype=np.float32))
    if pattern is not None:
        q = pattern.queries(q)
    return q.to(torch.bfloat16).to(device)


def make_latent(seed, B, T, device="cpu", amplitude=1.0):
    """New latents of T positions per request: bf16 [B, T, 576] ~ amplitude * N(0, 1)."""
    rng = np.random.default_rng([int(seed), 5])
    x = rng.standard_normal((B, T, D_QK), dtype=np.float32) * np.float32(amplitude)
    return torch.from_numpy(x).to(torch.bfloat16).to(device)


def make_decode_case(seed, lens, H, T=1, *, device="cpu", permute=True, max_pages=None,
                     extra_pages=0, kv_scale=None, sm_scale=SM_SCALE, pattern=None) -> DecodeCase:
    """Seeded decode inputs for contexts ``lens`` (each includes the T new positions).
    ``pattern``: an optional stress pattern (below) that reshapes the latents and
    queries before quantisation."""
    device = torch.device(device)
    lens = [int(x) for x in lens]
    padded = [((L + PAGE - 1) // PAGE) * PAGE for L in lens]
    if pattern is not None and kv_scale is None:
        kv_scale = pattern.fixed_scale()
    blocks, scale = _latent_codes(seed, padded, device, kv_scale, pattern)
    kv, bt = paginate(blocks, seed, device, permute=permute, max_pages=max_pages,
                      extra_pages=extra_pages)
    q = make_q(seed, len(lens), T, H, device, pattern)
    sl = torch.tensor(lens, dtype=torch.int32, device=device)
    ks = torch.tensor([scale], dtype=torch.float32, device=device)
    return DecodeCase(q, kv, ks, bt, sl, sm_scale, lens)


# ----------------------------------------------------------------------------
# Stress patterns: structured latents and queries that drive the softmax into
# its hard regimes (peaked, climbing, long flat tails far below a peak) while
# the values (latent dims [0, 512)) keep magnitudes where a bf16 answer can
# meet the absolute tolerance.  Structure is planted along one direction u
# spread evenly over the 64 positional dims [512, 576): a position's score
# then moves with its planted amplitude times the query's alignment with u.
# Input generation only: no attention arithmetic happens here.
# ----------------------------------------------------------------------------

def planted_direction(device="cpu"):
    """Unit vector with 1/8 in each of the 64 positional dims, 0 elsewhere."""
    u = torch.zeros(D_QK, dtype=torch.float32, device=device)
    u[D_V:] = 0.125
    return u


class StressPattern:
    """Base: N(0,1) latents and queries, unchanged."""

    def latents(self, b, c0, x):  # x: fp32 [m, 576] of positions c0 ..
        return x

    def queries(self, q):  # q: fp32 [B, T, H, 576]
        return q

    def fixed_scale(self):  # None: scale = amax / 448
        return None


class PeakedQueries(StressPattern):
    """Queries multiplied by ``gain``: scores gain times wider, a peaked softmax."""

    def __init__(self, gain):
        self.gain = float(gain)

    def queries(self, q):
        return q * self.gain


class ClimbingKeys(StressPattern):
    """Scores that climb: position p carries amplitude amp * ((p % period) + 1) / period
    along u, and the queries of heads h % 2 == 0 align with u with weight ``align``
    (the others keep N(0,1) queries, so both regimes share a call).  With a period
    equal to a partition's positions every partition's largest score sits on its
    last page and the running maximum moves again and again."""

    def __init__(self, amp, period, align=8.0, q_noise=1.0):
        self.amp, self.period, self.align, self.q_noise = float(amp), int(period), float(align), float(q_noise)

    def latents(self, b, c0, x):
        m = x.shape[0]
        p = torch.arange(c0, c0 + m, device=x.device, dtype=torch.float32)
        a = self.amp * (torch.remainder(p, self.period) + 1.0) / self.period
        return x + a[:, None] * planted_direction(x.device)[None, :]

    def queries(self, q):
        q = q * self.q_noise
        q[:, :, 0::2, :] += self.align * planted_direction()
        return q


class FirstPeak(StressPattern):
    """One dominant position: position 0 of every request carries amplitude ``amp``
    along u and every query is mostly u (noise ``q_noise``), so position 0 scores
    ``gap`` natural-log units or more above all others."""

    def __init__(self, amp, align=8.0, q_noise=0.05):
        self.amp, self.align, self.q_noise = float(amp), float(align), float(q_noise)

    def latents(self, b, c0, x):
        if c0 == 0:
            x = x.clone()
            x[0] += self.amp * planted_direction(x.device)
        return x

    def queries(self, q):
        return q * self.q_noise + self.align * planted_direction()


class CoherentTail(StressPattern):
    """The flush regime at its worst: position 0 of request b carries amplitude
    ``amps[b]`` along u; every other position holds the same latent (a fixed
    value vector with entries +-value, zero positional dims), so all of them
    score exactly the same, some distance below position 0, and their rounding
    errors add up coherently.  Queries are exactly ``align`` * u (zero value
    dims), so that distance is align * amps[b] * sm_scale (natural log units)."""

    def __init__(self, amps, align=8.0, value=1.0):
        self.amps, self.align, self.value = [float(a) for a in amps], float(align), float(value)

    def latents(self, b, c0, x):
        sign = torch.where(torch.arange(D_V, device=x.device) % 3 == 0, -1.0, 1.0)
        y = torch.zeros_like(x)
        y[:, :D_V] = self.value * sign[None, :]
        if c0 == 0:  # position 0: random values, positional dims exactly amp * u
            y[0, :D_V] = x[0, :D_V]
            y[0, D_V:] = self.amps[b % len(self.amps)] * planted_direction(x.device)[D_V:]
        return y

    def queries(self, q):
        return torch.zeros_like(q) + self.align * planted_direction()


class OutlierQueries(StressPattern):
    """One channel of every query row (a different one per row) ``ratio`` times the
    others' scale: the row is outlier * e_d + (outlier / ratio) * N(0,1), so the
    exact two-term query split must carry elements 2^-10 of the row's maximum
    (and below) while the scores stay of the usual size (outlier * x_d *
    sm_scale)."""

    def __init__(self, ratio=1024.0, outlier=16.0):
        self.ratio, self.outlier = float(ratio), float(outlier)

    def queries(self, q):
        B, T, H, D = q.shape
        q = q * (self.outlier / self.ratio)
        idx = (torch.arange(B * T * H) * 37) % D
        flat = q.view(-1, D)
        rows = torch.arange(B * T * H)
        flat[rows, idx] = torch.where(flat[rows, idx] >= 0, self.outlier, -self.outlier)
        return q


class ScaledCache(StressPattern):
    """Latents times ``latent_gain`` quantised with a fixed ``kv_scale`` (not
    amax / 448), and queries times ``q_gain``: a tiny scale with huge queries, or
    a large scale with codes in e4m3's subnormal range."""

    def __init__(self, latent_gain, kv_scale, q_gain):
        self.latent_gain, self.kv_scale, self.q_gain = float(latent_gain), float(kv_scale), float(q_gain)

    def latents(self, b, c0, x):
        return x * self.latent_gain

    def queries(self, q):
        return q * self.q_gain

    def fixed_scale(self):
        return self.kv_scale


@dataclass
class ShardedCase:
    """A history cut into contiguous shards, each paged on its own (DCP shape)."""
    shards: list          # DecodeCase per shard (shared q and kv_scale)
    full: DecodeCase      # the same history unsharded, for the oracle
    shard_len: int


def make_sharded_case(seed, B, H, total_len, n_shards, *, device="cpu", with_full=True, T=1):
    """Global history of ``total_len`` positions per request, one per-tensor scale
    over all of it, cut into ``n_shards`` contiguous shards of equal length.  With
    T > 1 the last T positions of the history are the draft positions of a
    multi-token verify (they fall in the last shard)."""
    device = torch.device(device)
    assert total_len % n_shards == 0
    sl = total_len // n_shards
    padded_full = [((total_len + PAGE - 1) // PAGE) * PAGE] * B
    blocks, scale = _latent_codes(seed, padded_full, device)
    q = make_q(seed, B, T, H, device)
    ks = torch.tensor([scale], dtype=torch.float32, device=device)
    shards = []
    spad = ((sl + PAGE - 1) // PAGE) * PAGE
    for s in range(n_shards):
        sb = []
        for b in range(B):
            blk = torch.zeros((spad, D_QK), dtype=torch.uint8, device=device)
            blk[:sl] = blocks[b][s * sl:(s + 1) * sl]
            sb.append(blk)
        kv, bt = paginate(sb, seed * 100 + s + 1, device)
        shards.append(DecodeCase(q, kv, ks, bt,
                                 torch.full((B,), sl, dtype=torch.int32, device=device),
                                 SM_SCALE, [sl] * B))
        del sb
    full = None
    if with_full:
        kv, bt = paginate(blocks, seed, device)
        full = DecodeCase(q, kv, ks, bt, torch.full((B,), total_len, dtype=torch.int32, device=device),
                          SM_SCALE, [total_len] * B)
    return ShardedCase(shards, full, sl)


# ----------------------------------------------------------------------------
# The five workloads (shapes, seeds and length mixes), full size and reduced.
# ----------------------------------------------------------------------------

def tp8_lens(seed, B=8, L=32768):
    return [L] * B


def verify_lens(seed, B=16, lo=8192, hi=131072):
    rng = np.random.default_rng([int(seed), 5])
    return [int(x) for x in rng.integers(lo, hi, size=B, endpoint=True)]


def ragged_lens(seed, B=128, lo=1024, hi=142000):
    rng = np.random.default_rng([int(seed), 5])
    u = rng.uniform(math.log(lo), math.log(hi), size=B)
    return [int(round(math.exp(x))) for x in u]


WORKLOADS = {
    # name: (description, seed)
    "tiny": ("1 request x 12 heads x 1 position, context 1024, n_splits=4", 1),
    "tp8_batch": ("8 requests x 12 heads x 1 position, context 32768 each", 2),
    "dcp_shard": ("32 requests x 96 heads x 1 position, 8 shards of 17,750 (142,000 total)", 3),
    "verify": ("16 requests x 12 heads x 4 causal positions, contexts U[8192,131072]", 4),
    "long": ("1 request x 12 heads x 1 position, context 393,216, auto splits", 5),
    "ragged": ("128 requests x 12 heads x 1 position, contexts log-U[1024,142000]", 6),
}


def workload_case(name, device="cpu", reduced=False, requests=0):
    """Inputs for one named workload; ``reduced`` shrinks contexts for the oracle;
    ``requests`` > 0 keeps the first that many requests of the batch (the same
    latents for them; a smaller case of the same shape)."""
    seed = WORKLOADS[name][1]

    def first(lens):
        return lens[:requests] if requests else lens

    if name == "tiny":
        return make_decode_case(seed, [1024], 12, 1, device=device)
    if name == "tp8_batch":
        L = 2 * 1024 + 37 if reduced else 32768
        return make_decode_case(seed, first(tp8_lens(seed, 8 if not reduced else 3, L)), 12, 1, device=device)
    if name == "verify":
        lens = verify_lens(seed, 4, 300, 1400) if reduced else verify_lens(seed)
        return make_decode_case(seed, first(lens), 12, 4, device=device)
    if name == "long":
        L = 20000 + 13 if reduced else 393216
        return make_decode_case(seed, [L], 12, 1, device=device)
    if name == "dcp_shard":  # one DCP shard as decoded locally: out + lse over its positions
        L = 300 + 11 if reduced else 17750
        return make_decode_case(seed, first([L] * (2 if reduced else 32)), 96, 1, device=device)
    if name == "ragged":
        lens = ragged_lens(seed, 16, 64, 3000) if reduced else ragged_lens(seed)
        return make_decode_case(seed, first(lens), 12, 1, device=device)
    raise KeyError(name)
