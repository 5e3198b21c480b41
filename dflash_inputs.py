"""Seeded synthetic inputs for the DFlash draft body and greedy verification.

This module is the only code shared by the CUDA path's callers (tests, bench) and the
fp64 oracle's callers.  It produces data and shapes only: it holds none of the method's
arithmetic (no projection, attention, normalisation, anchor choice or argmax).

Every tensor is drawn from its own NumPy PCG64 stream keyed by
(data seed, tensor id, indices), so any slice (one batch row, one chunk of context
positions, one draft layer) can be regenerated on its own without drawing the rest.
Floating-point values are sampled in float32 and rounded to bfloat16 with
round-to-nearest-even when the workload is bf16; both sides then see identical bits.

Workload shapes follow the configurations the DFlash pages describe:
* "angelspec DFlash" page, section "Configuration": hidden 4096, 5 draft layers,
  5 target layers of width 4096 taken at ids [1, 9, 17, 25, 33] of 36, vocab 151936;
  default block_size 16 (section "How it works").
* the Qwen3-8B-shaped attention sizes (32 query / 8 KV heads of width 128, SwiGLU 12288).
"""
from __future__ import annotations

import dataclasses
from dataclasses import dataclass, field

import numpy as np

# --------------------------------------------------------------------------------------
# shapes
# --------------------------------------------------------------------------------------


@dataclass(frozen=True)
class DraftShape:
    """Draft-body shape, mirroring the DFlash JSON config fields that fix tensor sizes."""

    target_hidden: int          # target_hidden_size (D_t)
    num_target_layers: int      # num_target_layers (n_tl); the concat width is n_tl * D_t
    hidden: int                 # hidden_size (D)
    num_layers: int             # num_hidden_layers of the draft (NL)
    num_heads: int              # query heads (Hq)
    num_kv_heads: int           # key/value heads (Hkv)
    head_dim: int               # dh
    intermediate: int           # SwiGLU width (I)
    rope_theta: float = 1.0e6
    rms_eps: float = 1.0e-6
    block_size: int = 16        # anchor + gamma draft positions (S = gamma + 1)
    dtype: str = "bf16"         # "bf16" or "f32": storage/arithmetic type of the path
    final_norm: bool = True
    ctx_norm: bool = True

    @property
    def concat_width(self) -> int:
        return self.num_target_layers * self.target_hidden

    @property
    def q_width(self) -> int:
        return self.num_heads * self.head_dim

    @property
    def kv_width(self) -> int:
        return self.num_kv_heads * self.head_dim

    @property
    def qkv_width(self) -> int:
        return self.q_width + 2 * self.kv_width


@dataclass(frozen=True)
class Workload:
    """One synthetic workload: shape + batch structure + verification inputs."""

    name: str
    index: int                  # data seed = 1000 + index
    shape: DraftShape
    batch: int                  # B (rows)
    seq_len: int                # L (target context length)
    num_anchors: int            # N anchors per row
    # rows whose mask is right-padded: (row, valid_length)
    padded_rows: tuple = ()
    # groups of rows that share a sample id (and identical masks / hidden states)
    shared_sid_groups: tuple = ()
    # inference layout: one block per row, anchor fixed at seq_len (the cached context)
    inference: bool = False
    # greedy verification inputs
    verify_batch: int = 0
    vocab: int = 0
    verify_dtype: str = "bf16"
    verify_accept_p: float = 0.3   # geometric(p) accepted-prefix length
    plan_seed: int = 0xD1F1A5
    plan_step: int = 0

    @property
    def data_seed(self) -> int:
        return 1000 + self.index

    @property
    def tokens(self) -> int:
        """Planned draft slots T = B * N * S (the metric's block positions per step)."""
        return self.batch * self.num_anchors * self.shape.block_size


TINY_F32 = DraftShape(target_hidden=256, num_target_layers=2, hidden=256, num_layers=1,
                      num_heads=4, num_kv_heads=2, head_dim=64, intermediate=512,
                      block_size=4, dtype="f32")

QWEN3_8B_DRAFT = DraftShape(target_hidden=4096, num_target_layers=5, hidden=4096,
                            num_layers=5, num_heads=32, num_kv_heads=8, head_dim=128,
                            intermediate=12288, block_size=16, dtype="bf16")


def _workloads() -> dict:
    w = {}
    w["tiny_f32"] = Workload("tiny_f32", 0, TINY_F32, batch=1, seq_len=128, num_anchors=4,
                             verify_batch=4, vocab=1000, verify_dtype="f32")
    w["train_8b_b4_l2048"] = Workload("train_8b_b4_l2048", 1, QWEN3_8B_DRAFT, batch=4,
                                      seq_len=2048, num_anchors=8, padded_rows=((3, 1),),
                                      verify_batch=32, vocab=151936)
    for i, b in enumerate((1, 8, 32, 64)):
        name = f"decode_8b_b{b}_ctx4096"
        w[name] = Workload(name, 2, QWEN3_8B_DRAFT, batch=b, seq_len=4096, num_anchors=1,
                           inference=True, verify_batch=b, vocab=151936)
    w["longctx_8b_l32768"] = Workload("longctx_8b_l32768", 3, QWEN3_8B_DRAFT, batch=1,
                                      seq_len=32768, num_anchors=64)
    w["train_8b_b16_l4096"] = Workload("train_8b_b16_l4096", 4, QWEN3_8B_DRAFT, batch=16,
                                       seq_len=4096, num_anchors=32,
                                       shared_sid_groups=((0, 1), (2, 3), (4, 5), (6, 7)))
    return w


WORKLOADS = _workloads()


def smoke_workload() -> Workload:
    """A small bf16 case of the whole path (several tiles in the GEMMs, one right-padded
    row, a key range of one chunk, 24 draft slots) plus verification over a vocab of 5000."""
    shape = DraftShape(target_hidden=128, num_target_layers=2, hidden=256, num_layers=2,
                       num_heads=4, num_kv_heads=2, head_dim=128, intermediate=384,
                       block_size=4, dtype="bf16")
    return Workload("smoke", 9, shape, batch=2, seq_len=160, num_anchors=3,
                    padded_rows=((1, 90),), verify_batch=3, vocab=5000)


def scaled(w: Workload, **kw) -> Workload:
    """A copy of a workload with some fields (or shape fields) replaced; for small tests."""
    shape_kw = {k: kw.pop(k) for k in list(kw) if k in DraftShape.__dataclass_fields__}
    shape = dataclasses.replace(w.shape, **shape_kw) if shape_kw else w.shape
    return dataclasses.replace(w, shape=shape, **kw)


# --------------------------------------------------------------------------------------
# bit-level helpers (data representation only)
# --------------------------------------------------------------------------------------


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 to bfloat16 (round-to-nearest-even); returns uint16 bit patterns.

    Inputs here are finite samples, so no NaN handling is needed.
    """
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    bias = ((u >> np.uint32(16)) & np.uint32(1)) + np.uint32(0x7FFF)
    return ((u + bias) >> np.uint32(16)).astype(np.uint16)


def bf16_bits_to_f64(b: np.ndarray) -> np.ndarray:
    """Exact widening of bfloat16 bit patterns to float64."""
    return (b.astype(np.uint32) << np.uint32(16)).view(np.float32).astype(np.float64)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    return (b.astype(np.uint32) << np.uint32(16)).view(np.float32)


class Tensor:
    """A synthetic tensor in its storage form ("bf16" uint16 bits or "f32" float32)."""

    __slots__ = ("data", "dtype")

    def __init__(self, data: np.ndarray, dtype: str):
        self.data = data
        self.dtype = dtype

    @property
    def shape(self):
        return self.data.shape

    def f64(self) -> np.ndarray:
        if self.dtype == "bf16":
            return bf16_bits_to_f64(self.data)
        return self.data.astype(np.float64)

    def f32(self) -> np.ndarray:
        if self.dtype == "bf16":
            return bf16_bits_to_f32(self.data)
        return self.data.astype(np.float32)


# tensor ids of the per-tensor streams
_ID = {"w_proj": 1, "g_ctx": 2, "g_final": 3, "g_in": 10, "w_qkv": 11, "w_o": 12,
       "g_post": 13, "w_gate_up": 14, "w_down": 15, "hidden": 20, "emb": 21, "sid": 22,
       "logits": 30, "draft": 31, "accept": 32, "plant": 33, "lm_head": 40, "targets": 41}

HIDDEN_CHUNK = 256  # positions per independent stream of target hidden states


def _rng(*key: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(np.random.SeedSequence(list(key))))


def _normal(rng: np.random.Generator, shape, std: float, dtype: str) -> Tensor:
    x = rng.standard_normal(size=shape, dtype=np.float32)
    if std != 1.0:
        x *= np.float32(std)
    if dtype == "bf16":
        return Tensor(f32_to_bf16_bits(x), "bf16")
    return Tensor(x, "f32")


# --------------------------------------------------------------------------------------
# weights
# --------------------------------------------------------------------------------------


def gen_top_weights(w: Workload, gain_std: float = 0.0) -> dict:
    """W_proj [D, n_tl*D_t] (rows = outputs), g_ctx [D], g_final [D]."""
    s = w.shape
    out = {"w_proj": _normal(_rng(w.data_seed, _ID["w_proj"]), (s.hidden, s.concat_width),
                             0.02, s.dtype)}
    for name in ("g_ctx", "g_final"):
        out[name] = _gain(w, name, 0, gain_std)
    return out


def _gain(w: Workload, name: str, layer: int, gain_std: float) -> Tensor:
    s = w.shape
    if gain_std == 0.0:
        g = np.ones(s.hidden, np.float32)
    else:
        g = 1.0 + gain_std * _rng(w.data_seed, _ID[name], layer).standard_normal(
            s.hidden, dtype=np.float32)
    if s.dtype == "bf16":
        return Tensor(f32_to_bf16_bits(g), "bf16")
    return Tensor(g.astype(np.float32), "f32")


def gen_layer_weights(w: Workload, layer: int, gain_std: float = 0.0) -> dict:
    """One draft decoder layer, every matrix stored [out_features, in_features]:

    w_qkv [Hq*dh + 2*Hkv*dh, D]  (rows: all Q heads, then all K heads, then all V heads)
    w_o [D, Hq*dh], w_gate_up [2*I, D] (rows: I gate rows, then I up rows), w_down [D, I].
    """
    s = w.shape
    seed = w.data_seed
    return {
        "g_in": _gain(w, "g_in", layer, gain_std),
        "w_qkv": _normal(_rng(seed, _ID["w_qkv"], layer), (s.qkv_width, s.hidden), 0.02, s.dtype),
        "w_o": _normal(_rng(seed, _ID["w_o"], layer), (s.hidden, s.q_width), 0.02, s.dtype),
        "g_post": _gain(w, "g_post", layer, gain_std),
        "w_gate_up": _normal(_rng(seed, _ID["w_gate_up"], layer), (2 * s.intermediate, s.hidden),
                             0.02, s.dtype),
        "w_down": _normal(_rng(seed, _ID["w_down"], layer), (s.hidden, s.intermediate), 0.02,
                          s.dtype),
    }


# --------------------------------------------------------------------------------------
# batch structure
# --------------------------------------------------------------------------------------


def source_row(w: Workload, b: int) -> int:
    """Rows in a shared-sample-id group carry the first row's data (identical inputs)."""
    for grp in w.shared_sid_groups:
        if b in grp:
            return min(grp)
    return b


def gen_mask(w: Workload) -> np.ndarray:
    """Input mask [B, L] uint8: 1 = valid target position.  Padded rows are right-padded."""
    m = np.ones((w.batch, w.seq_len), np.uint8)
    for row, valid_len in w.padded_rows:
        m[row, valid_len:] = 0
    return m


def gen_sample_ids(w: Workload) -> np.ndarray:
    """Distinct random int64 sample ids, shared within each shared-sid group."""
    rng = _rng(w.data_seed, _ID["sid"])
    ids = rng.integers(-(2 ** 62), 2 ** 62, size=w.batch, dtype=np.int64)
    out = ids.copy()
    for b in range(w.batch):
        out[b] = ids[source_row(w, b)]
    return out


def gen_target_hidden_rows(w: Workload, b: int, c0: int, c1: int) -> Tensor:
    """Concatenated selected target hidden states for row b, positions [c0, c1):
    shape [c1 - c0, n_tl * D_t], N(0, 1).  Generated in chunks of HIDDEN_CHUNK positions
    so that any range is reproducible on its own."""
    s = w.shape
    src = source_row(w, b)
    parts = []
    k0, k1 = c0 // HIDDEN_CHUNK, (c1 + HIDDEN_CHUNK - 1) // HIDDEN_CHUNK
    for k in range(k0, k1):
        n = min(HIDDEN_CHUNK, w.seq_len - k * HIDDEN_CHUNK)
        t = _normal(_rng(w.data_seed, _ID["hidden"], src, k), (n, s.concat_width), 1.0, s.dtype)
        lo = max(c0 - k * HIDDEN_CHUNK, 0)
        hi = min(c1 - k * HIDDEN_CHUNK, n)
        parts.append(t.data[lo:hi])
    return Tensor(np.concatenate(parts, axis=0), s.dtype)


def _parallel(fn, items) -> None:
    """Runs fn over items on a few threads (NumPy's generators release the GIL while they
    fill large arrays); the values do not depend on the thread count or order."""
    import concurrent.futures as cf
    import os
    items = list(items)
    n = min(len(items), os.cpu_count() or 1, 16)
    if n <= 1:
        for it in items:
            fn(it)
        return
    with cf.ThreadPoolExecutor(max_workers=n) as ex:
        list(ex.map(fn, items))


def gen_target_hidden(w: Workload) -> Tensor:
    """All rows: [B, L, n_tl * D_t]."""
    s = w.shape
    dt = np.uint16 if s.dtype == "bf16" else np.float32
    out = np.empty((w.batch, w.seq_len, s.concat_width), dt)
    chunks = (w.seq_len + HIDDEN_CHUNK - 1) // HIDDEN_CHUNK

    def fill(item):
        b, k = item
        c0, c1 = k * HIDDEN_CHUNK, min(w.seq_len, (k + 1) * HIDDEN_CHUNK)
        out[b, c0:c1] = gen_target_hidden_rows(w, b, c0, c1).data
    _parallel(fill, [(b, k) for b in range(w.batch) for k in range(chunks)])
    return Tensor(out, s.dtype)


def gen_block_emb(w: Workload) -> Tensor:
    """Caller-supplied embeddings for every block slot [B, N, S, D], iid N(0, 1)."""
    s = w.shape
    dt = np.uint16 if s.dtype == "bf16" else np.float32
    out = np.empty((w.batch, w.num_anchors, s.block_size, s.hidden), dt)
    for b in range(w.batch):
        t = _normal(_rng(w.data_seed, _ID["emb"], source_row(w, b)),
                    (w.num_anchors, s.block_size, s.hidden), 1.0, s.dtype)
        out[b] = t.data
    return Tensor(out, s.dtype)


def inference_block_layout(w: Workload):
    """Inference layout: each row has one block whose anchor sits right after the cached
    context (anchor = L), every slot valid, positions L .. L + S - 1."""
    S = w.shape.block_size
    anchors = np.full((w.batch, 1), w.seq_len, np.int32)
    block_valid = np.ones((w.batch, 1, S), np.uint8)
    position_ids = (w.seq_len + np.arange(S, dtype=np.int32))[None, None, :].repeat(w.batch, 0)
    return anchors, block_valid, position_ids.astype(np.int32)


# --------------------------------------------------------------------------------------
# verification inputs
# --------------------------------------------------------------------------------------


@dataclass
class VerifyInputs:
    logits: Tensor                 # [Bv, S, V]
    draft: np.ndarray              # int32 [Bv, S - 1]
    eos: int                       # -1 = none
    planted_prefix: np.ndarray     # int32 [Bv]: drafts agree with the planted maxima up to here
    planted_top: np.ndarray = field(default=None)  # int32 [Bv, S]: planted maximum per position


PLANT_VALUE = 8.0   # exactly representable in bf16; far above any N(0,1) draw at V <= 2^20


def gen_verify(w: Workload, batch: int | None = None, eos: int = -1) -> VerifyInputs:
    """Target logits N(0,1) [Bv, S, V] with one planted maximum per position, and draft
    tokens that follow the planted maxima for a geometric(p) prefix length G (capped at
    gamma), then differ at position G.

    The planted maximum (value PLANT_VALUE at a random token) makes the intended argmax
    known by construction, without computing one here."""
    S = w.shape.block_size
    gamma = S - 1
    Bv = w.verify_batch if batch is None else batch
    V = w.vocab
    bf16 = w.verify_dtype == "bf16"
    x = np.empty((Bv, S, V), np.float32)
    out = np.empty((Bv, S, V), np.uint16) if bf16 else x

    def fill(b):  # one stream per request
        x[b] = _rng(w.data_seed, _ID["logits"], Bv, b).standard_normal(size=(S, V),
                                                                        dtype=np.float32)
    _parallel(fill, range(Bv))
    prng = _rng(w.data_seed, _ID["plant"], Bv)
    top = prng.integers(0, V, size=(Bv, S), dtype=np.int64).astype(np.int32)
    x[np.arange(Bv)[:, None], np.arange(S)[None, :], top] = PLANT_VALUE
    arng = _rng(w.data_seed, _ID["accept"], Bv)
    g = arng.geometric(w.verify_accept_p, size=Bv) - 1
    k = np.minimum(g, gamma).astype(np.int32)
    drng = _rng(w.data_seed, _ID["draft"], Bv)
    draft = drng.integers(0, V, size=(Bv, gamma), dtype=np.int64).astype(np.int32)
    for b in range(Bv):
        draft[b, :k[b]] = top[b, :k[b]]
        if k[b] < gamma and draft[b, k[b]] == top[b, k[b]]:
            draft[b, k[b]] = (top[b, k[b]] + 1) % V
    if bf16:
        def conv(b):
            out[b] = f32_to_bf16_bits(x[b])
        _parallel(conv, range(Bv))
        lt = Tensor(out, "bf16")
    else:
        lt = Tensor(x, "f32")
    return VerifyInputs(lt, draft, eos, k, top)


# --------------------------------------------------------------------------------------
# draft loss inputs
# --------------------------------------------------------------------------------------

LM_CHUNK = 8192  # vocab rows per independent stream of the lm_head


def gen_lm_head(w: Workload, vocab: int) -> Tensor:
    """A frozen lm_head stand-in [V, D], iid N(0, 0.02) in the workload's dtype."""
    s = w.shape
    dt = np.uint16 if s.dtype == "bf16" else np.float32
    out = np.empty((vocab, s.hidden), dt)

    def fill(k):
        r0, r1 = k * LM_CHUNK, min(vocab, (k + 1) * LM_CHUNK)
        out[r0:r1] = _normal(_rng(w.data_seed, _ID["lm_head"], k), (r1 - r0, s.hidden), 0.02,
                             s.dtype).data
    _parallel(fill, range((vocab + LM_CHUNK - 1) // LM_CHUNK))
    return Tensor(out, s.dtype)


def gen_targets(w: Workload, vocab: int) -> np.ndarray:
    """Ground-truth token of every block slot [B, N, S] int32, uniform over the vocab."""
    rng = _rng(w.data_seed, _ID["targets"])
    return rng.integers(0, vocab, size=(w.batch, w.num_anchors, w.shape.block_size),
                        dtype=np.int64).astype(np.int32)

