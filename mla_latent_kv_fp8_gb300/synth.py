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


def _latent_codes(seed, lens_padded, device, scale=None):
    """Per-request FP8 code blocks [Lpad_b, 576] for N(0,1) latents.

    Two passes over the same seed-addressed chunks: amax first (unless a scale
    is supplied), then quantisation.  Returns (list of uint8 tensors, scale)."""
    chunk = _CHUNK_CUDA if device.type == "cuda" else _CHUNK
    if scale is None:
        amax = 0.0
        for b, L in enumerate(lens_padded):
            for c0 in range(0, L, chunk):
                n = min(chunk, L - c0) * D_QK
                x = _normal_chunk((seed, 7, b, c0), n, device)
                amax = max(amax, float(x.abs().max()))
        scale = np.float32(amax) / np.float32(FP8_MAX)
    scale = np.float32(scale)
    blocks = []
    st = torch.tensor(float(scale), dtype=torch.float32, device=device)
    for b, L in enumerate(lens_padded):
        out = torch.empty((L, D_QK), dtype=torch.uint8, device=device)
        for c0 in range(0, L, chunk):
            m = min(chunk, L - c0)
            x = _normal_chunk((seed, 7, b, c0), m * D_QK, device)
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


def make_q(seed, B, T, H, device="cpu"):
    rng = np.random.default_rng([int(seed), 3])
    q = torch.from_numpy(rng.standard_normal((B, T, H, D_QK), dtype=np.float32))
    return q.to(torch.bfloat16).to(device)


def make_latent(seed, B, T, device="cpu", amplitude=1.0):
    """New latents of T positions per request: bf16 [B, T, 576] ~ amplitude * N(0, 1)."""
    rng = np.random.default_rng([int(seed), 5])
    x = rng.standard_normal((B, T, D_QK), dtype=np.float32) * np.float32(amplitude)
    return torch.from_numpy(x).to(torch.bfloat16).to(device)


def make_decode_case(seed, lens, H, T=1, *, device="cpu", permute=True, max_pages=None,
                     extra_pages=0, kv_scale=None, sm_scale=SM_SCALE) -> DecodeCase:
    """Seeded decode inputs for contexts ``lens`` (each includes the T new positions)."""
    device = torch.device(device)
    lens = [int(x) for x in lens]
    padded = [((L + PAGE - 1) // PAGE) * PAGE for L in lens]
    blocks, scale = _latent_codes(seed, padded, device, kv_scale)
    kv, bt = paginate(blocks, seed, device, permute=permute, max_pages=max_pages,
                      extra_pages=extra_pages)
    q = make_q(seed, len(lens), T, H, device)
    sl = torch.tensor(lens, dtype=torch.int32, device=device)
    ks = torch.tensor([scale], dtype=torch.float32, device=device)
    return DecodeCase(q, kv, ks, bt, sl, sm_scale, lens)


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


def workload_case(name, device="cpu", reduced=False):
    """Inputs for one named workload; ``reduced`` shrinks contexts for the oracle."""
    seed = WORKLOADS[name][1]
    if name == "tiny":
        return make_decode_case(seed, [1024], 12, 1, device=device)
    if name == "tp8_batch":
        L = 2 * 1024 + 37 if reduced else 32768
        return make_decode_case(seed, tp8_lens(seed, 8 if not reduced else 3, L), 12, 1, device=device)
    if name == "verify":
        lens = verify_lens(seed, 4, 300, 1400) if reduced else verify_lens(seed)
        return make_decode_case(seed, lens, 12, 4, device=device)
    if name == "long":
        L = 20000 + 13 if reduced else 393216
        return make_decode_case(seed, [L], 12, 1, device=device)
    if name == "dcp_shard":  # one DCP shard as decoded locally: out + lse over its positions
        L = 300 + 11 if reduced else 17750
        return make_decode_case(seed, [L] * (2 if reduced else 32), 96, 1, device=device)
    if name == "ragged":
        lens = ragged_lens(seed, 16, 64, 3000) if reduced else ragged_lens(seed)
        return make_decode_case(seed, lens, 12, 1, device=device)
    raise KeyError(name)
