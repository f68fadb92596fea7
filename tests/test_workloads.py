"""The seeded input generators (no GPU): determinism, structure, and the five workloads' shapes."""
import numpy as np
import pytest

import workloads as W


def test_normal_bits_deterministic_and_unit_variance():
    a = W.normal_bits(3_000_000, "bf16", seed=5, stream=1, threads=4)
    b = W.normal_bits(3_000_000, "bf16", seed=5, stream=1, threads=1)
    c = W.normal_bits(3_000_000, "bf16", seed=6, stream=1)
    assert np.array_equal(a, b) and not np.array_equal(a, c)
    x = (a.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    assert abs(x.mean()) < 5e-3 and abs(x.var() - 1.0) < 5e-3
    h = W.normal_bits(1_000_000, "f16", seed=1).view(np.float16).astype(np.float64)
    assert abs(h.mean()) < 5e-3 and abs(h.var() - 1.0) < 5e-3


def test_allocator():
    al = W.BlockAllocator(10, np.random.default_rng(0))
    a = al.alloc(4)
    assert len(set(a)) == 4 and al.num_free == 6
    al.share(a[:2])
    al.free(a)
    assert al.num_free == 8 and list(al.refcount[a[:2]]) == [1, 1]
    al.free(a[:2])
    assert al.num_free == 10
    with pytest.raises(ValueError):
        al.free(a[:1])
    with pytest.raises(MemoryError):
        al.alloc(11)


def _check_decode(c: W.DecodeCase):
    bs = c.block_size
    used = []
    for i in range(c.B):
        n = int(c.context_lens[i])
        nb = (n + bs - 1) // bs
        row = c.block_tables[i]
        assert (row[:nb] >= 0).all() and (row[:nb] < c.num_blocks).all()
        assert (row[nb:] == -1).all()
        used += list(row[:nb])
        if c.slot_mapping[i] >= 0:
            p = n - 1
            assert c.slot_mapping[i] == row[p // bs] * bs + p % bs
    assert len(used) == len(set(used)), "decode sequences never share blocks"
    s = c.slot_mapping[c.slot_mapping >= 0]
    assert len(s) == len(set(s.tolist()))
    assert c.k_cache.shape == (c.num_blocks, bs, c.Hkv, c.D) == c.v_cache.shape
    assert c.q.shape == (c.B, c.Hq, c.D) and c.k_new.shape == (c.B, c.Hkv, c.D)
    return used


def test_tiny_config():
    c = W.make("tiny")
    assert list(c.context_lens) == [1, 17, 100, 255]
    assert (c.B, c.Hq, c.Hkv, c.D, c.block_size, c.num_blocks, c.dtype) == (4, 4, 2, 64, 16, 64, "f16")
    used = _check_decode(c)
    assert len(used) == 1 + 2 + 7 + 16
    assert c.scale == 1 / 8
    assert np.array_equal(W.make("tiny").k_cache, c.k_cache)


@pytest.mark.parametrize("name,lo,hi", [("qwen25_05b_decode", 128, 2048),
                                        ("qwen3_06b_decode", 100, 4096)])
def test_uniform_decode_configs(name, lo, hi):
    c = W.make(name, n=12)
    assert c.context_lens.min() >= lo and c.context_lens.max() <= hi
    used = _check_decode(c)
    assert c.num_blocks == int(np.ceil(1.25 * len(used)))
    assert c.max_blocks_per_seq * c.block_size == hi


def test_longtail_config_structure():
    lens = W._lengths("longtail_decode", W.CONFIGS["longtail_decode"].seed)
    assert len(lens) == 512 and lens.min() >= 1 and lens.max() <= 16384
    assert 1500 < np.median(lens) < 2800           # median 2048 by construction
    c = W.make("longtail_decode", n=24)
    used = _check_decode(c)
    assert len(used) / c.num_blocks >= 0.94        # pool near full
    gaps = [abs(int(r[1]) - int(r[0])) for r in c.block_tables if r[1] >= 0]
    assert np.mean(gaps) > 2                      # a sequence's blocks are scattered


def test_prefill_config_structure():
    c = W.make("prefill_prefix", n=6)
    assert (c.k_lens - c.q_lens == 512).all()
    assert c.q_lens.min() >= 100 and c.q_lens.max() <= 1024
    pre = c.block_tables[:, :2]
    assert (pre == pre[0]).all()                    # every prompt points at the same 2 blocks
    assert list(c.refcount[pre[0]]) == [6, 6]
    slots = c.slot_mapping
    assert len(set(slots.tolist())) == len(slots)
    assert not (np.isin(slots // c.block_size, pre[0])).any()
    for s in range(c.S):
        for r in (0, int(c.q_lens[s]) - 1):
            p = 512 + r
            assert slots[c.cu_seqlens_q[s] + r] == c.block_tables[s, p // 256] * 256 + p % 256


def test_qwen25_prefill_config_structure():
    """The Qwen2.5-shaped prefill: the prefill_prefix prompt mix at 14/2 heads, D 64, 16-token
    blocks, fp16; the shared 512-token prefix is 32 blocks every prompt points at."""
    c = W.make("qwen25_prefill", n=5)
    assert (c.Hq, c.Hkv, c.D, c.block_size, c.dtype) == (14, 2, 64, 16, "f16")
    assert (c.k_lens - c.q_lens == 512).all()
    assert c.q_lens.min() >= 100 and c.q_lens.max() <= 1024
    pre = c.block_tables[:, :32]
    assert (pre == pre[0]).all() and len(set(pre[0].tolist())) == 32
    assert (c.refcount[pre[0]] == 5).all()
    slots = c.slot_mapping
    assert len(set(slots.tolist())) == len(slots)
    assert not (np.isin(slots // c.block_size, pre[0])).any()
    for s in range(c.S):
        for r in (0, int(c.q_lens[s]) - 1):
            p = 512 + r
            assert slots[c.cu_seqlens_q[s] + r] == c.block_tables[s, p // 16] * 16 + p % 16
    assert np.array_equal(W.lengths("qwen25_prefill"), W.lengths("prefill_prefix", seed=5))
