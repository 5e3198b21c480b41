"""GPU greedy verification vs the oracle: bit-exact choices, emitted tokens and counts."""
import numpy as np
import pytest

import dflash_inputs as di
from oracle import dflash_oracle as orc

pytestmark = pytest.mark.gpu


def gpu_verify(logits: di.Tensor, draft: np.ndarray, eos: int = -1):
    import torch
    import block_draft_model_proj_gb300 as dflash
    from dflash_testlib import to_device
    B, S, V = logits.shape
    gamma = S - 1
    dl = to_device(logits)
    dd = torch.from_numpy(np.ascontiguousarray(draft, np.int32)).cuda()
    em = torch.full((B, S), -9, dtype=torch.int32, device="cuda")
    ne = torch.full((B,), -9, dtype=torch.int32, device="cuda")
    ac = torch.full((B,), -9, dtype=torch.int32, device="cuda")
    ch = torch.full((B, S), -9, dtype=torch.int32, device="cuda")
    dt = dflash.DFLASH_DTYPE_BF16 if logits.dtype == "bf16" else dflash.DFLASH_DTYPE_F32
    dflash.dflash_verify_greedy(dl, dt, dd, B, gamma, V, eos, em, ne, ac, ch)
    dflash.dflash_device_status()
    return ch.cpu().numpy(), em.cpu().numpy(), ne.cpu().numpy(), ac.cpu().numpy()


def check(logits: di.Tensor, draft, eos=-1):
    got = gpu_verify(logits, draft, eos)
    ref = orc.verify_greedy(logits.f64(), draft, eos)
    for g, r, name in zip(got, ref, ("choices", "emitted", "num_emitted", "accepted")):
        assert np.array_equal(g, r), name
    return got


def test_tiny_f32_config(lib):
    w = di.WORKLOADS["tiny_f32"]
    vi = di.gen_verify(w)
    ch, em, ne, ac = check(vi.logits, vi.draft)
    assert np.array_equal(ac, vi.planted_prefix)
    assert np.array_equal(ch, vi.planted_top)


@pytest.mark.parametrize("batch", [1, 8, 32, 64])
def test_decode_config_bf16(lib, batch):
    w = di.WORKLOADS[f"decode_8b_b{batch}_ctx4096"]
    vi = di.gen_verify(w)
    ch, em, ne, ac = check(vi.logits, vi.draft)
    assert np.array_equal(ac, vi.planted_prefix)
    # all-match rows emit the bonus
    for b in range(batch):
        if ac[b] == w.shape.block_size - 1:
            assert ne[b] == w.shape.block_size and em[b, -1] == ch[b, -1]


def test_pages_worked_example(lib):
    # draft [10, 20, 99, 40] against target choices [10, 20, 30, 40, 50]
    V = 64
    x = np.zeros((1, 5, V), np.float32)
    for i, t in enumerate([10, 20, 30, 40, 50]):
        x[0, i, t] = 1.0
    logits = di.Tensor(di.f32_to_bf16_bits(x), "bf16")
    ch, em, ne, ac = check(logits, np.array([[10, 20, 99, 40]], np.int32))
    assert list(em[0][:ne[0]]) == [10, 20, 30] and ac[0] == 2


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_ties_take_lowest_index(lib, dtype):
    rng = np.random.default_rng(31)
    B, S, V = 7, 5, 20011          # V odd: no 16-byte vector path
    x = rng.integers(-2, 3, size=(B, S, V)).astype(np.float32)   # many exact ties
    t = di.Tensor(di.f32_to_bf16_bits(x), "bf16") if dtype == "bf16" else di.Tensor(x, "f32")
    draft = rng.integers(0, 3, size=(B, S - 1)).astype(np.int32)
    ch, *_ = check(t, draft)
    assert np.all(ch < 50)   # ties resolve to early indices


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_ties_take_lowest_index_vector_path(lib, dtype):
    """Exact ties across 16-byte vectors, threads and vocab chunks (V a multiple of 8), and a
    row whose maximum is -inf everywhere."""
    rng = np.random.default_rng(37)
    B, S, V = 3, 4, 151936
    x = rng.integers(-2, 3, size=(B, S, V)).astype(np.float32)
    x[1, 2, :] = -np.inf
    x[2, 1, :] = -2.0
    x[2, 1, V - 5] = -1.0                     # a lone maximum near the end
    t = di.Tensor(di.f32_to_bf16_bits(x), "bf16") if dtype == "bf16" else di.Tensor(x, "f32")
    draft = rng.integers(0, 3, size=(B, S - 1)).astype(np.int32)
    ch, *_ = check(t, draft)
    assert ch[1, 2] == 0 and ch[2, 1] == V - 5


@pytest.mark.parametrize("V", [1, 7, 8, 4096, 151936, 262144 + 3])
def test_vocab_sizes_and_chunking(lib, V):
    rng = np.random.default_rng(V)
    B, S = 3, 4
    x = rng.standard_normal((B, S, V)).astype(np.float32)
    draft = rng.integers(0, V, size=(B, S - 1)).astype(np.int32)
    check(di.Tensor(di.f32_to_bf16_bits(x), "bf16"), draft)
    check(di.Tensor(x, "f32"), draft)


def test_eos_and_gamma_zero(lib):
    V = 32
    x = np.zeros((3, 4, V), np.float32)
    choices = [[5, 0, 7, 9], [5, 6, 7, 9], [5, 6, 7, 9]]
    for b in range(3):
        for i, c in enumerate(choices[b]):
            x[b, i, c] = 2.0
    logits = di.Tensor(di.f32_to_bf16_bits(x), "bf16")
    draft = np.array([[5, 0, 7], [5, 6, 7], [5, 1, 7]], np.int32)
    ch, em, ne, ac = check(logits, draft, eos=0)
    assert list(em[0][:ne[0]]) == [5, 0] and ac[0] == 2        # EOS accepted: no bonus
    assert list(em[1][:ne[1]]) == [5, 6, 7, 9] and ac[1] == 3   # bonus
    assert list(em[2][:ne[2]]) == [5, 6] and ac[2] == 1
    # gamma = 0: only the bonus is emitted
    ch, em, ne, ac = check(di.Tensor(di.f32_to_bf16_bits(x[:, :1]), "bf16"),
                           np.zeros((3, 0), np.int32))
    assert np.all(ne == 1) and np.all(ac == 0) and list(em[:, 0]) == [5, 5, 5]
