"""The host block manager (pa_bm_*) against the reference model in oracle/block_manager.py.

The model is pinned first by hand-worked scenarios (expected block ids, hits and reference counts
derived from the rules the model's docstring states). The library is then driven with seeded
random workloads (prompts that share system-prompt prefixes, decode appends, finishes,
preemptions that release and re-admit a sequence with its tokens, a pool under pressure) and must
agree with the model on every returned value and on the whole state after every operation. With
the test-only degenerate hash every token hash collides: the library may then miss hits the model
finds, but every hit it takes must still be exact.
"""
import numpy as np
import pytest

from oracle.block_manager import BlockManagerModel, NoBlocks
from paged_kv_cache_83_gb300 import binding
import paged_kv_cache_83_gb300 as pa


@pytest.fixture(scope="module", autouse=True)
def lib():
    if not binding.LIB_PATH.exists():
        from paged_kv_cache_83_gb300 import build
        build.build()
    return pa.load()


# ------------------------------------------------------------------------------------------
# the model, pinned by hand
# ------------------------------------------------------------------------------------------

def test_model_first_sequence_takes_blocks_in_id_order():
    m = BlockManagerModel(8, 4)
    assert m.allocate("a", range(1, 10)) == 0          # 9 tokens: 3 blocks, nothing cached
    assert m.table("a") == [0, 1, 2] and m.num_free() == 5
    assert m.ref[:4] == [1, 1, 1, 0]


def test_model_shared_prefix_but_never_the_last_tokens_block():
    m = BlockManagerModel(8, 4)
    m.allocate("a", range(1, 10))                      # blocks 0 [1-4], 1 [5-8], 2 [9]
    assert m.allocate("b", range(1, 11)) == 8          # [1-4], [5-8] reused, [9,10] new
    assert m.table("b") == [0, 1, 3] and m.ref[:4] == [2, 2, 1, 1]
    # exactly two full blocks: the second holds the last token, so only the first is reused
    assert m.allocate("c", range(1, 9)) == 4
    assert m.table("c") == [0, 4] and m.ref[0] == 3


def test_model_release_and_free_queue_order():
    m = BlockManagerModel(4, 2)
    m.allocate("a", [1, 2, 3, 4, 5])                   # blocks 0, 1, 2
    m.release("a")                                     # last block first: queue 3, 2, 1, 0
    assert m.free == [3, 2, 1, 0] and m.ref == [0, 0, 0, 0]
    # the cached prefix is found again and leaves the middle of the queue
    assert m.allocate("b", [1, 2, 3, 4, 9]) == 4
    assert m.table("b") == [0, 1, 3] and m.free == [2]


def test_model_taking_a_block_forgets_it_and_its_children():
    m = BlockManagerModel(3, 2)
    m.allocate("a", [1, 2, 3, 4, 5])                   # 0 [1,2], 1 [3,4] (parent 0), 2 [5]
    m.release("a")                                     # queue 2, 1, 0
    m.allocate("x", [7, 7, 7, 7, 7, 7])                # takes 2, 1, 0 for new content
    m.release("x")                                     # queue 0, 1, 2
    # [1,2] and [3,4] are gone (blocks reused); [7,7],[7,7] chain is cached
    assert m.allocate("b", [1, 2, 3, 4, 5]) == 0
    m.release("b")
    assert m.allocate("c", [1, 2, 3, 4, 6]) == 4       # b's blocks are cached now


def test_model_append_caches_filled_blocks():
    m = BlockManagerModel(6, 2)
    m.allocate("a", [1])
    assert m.append("a", 2) == 1                       # slot 0 * 2 + 1
    assert m.append("a", 3) == 2 * 1 + 0               # new block 1
    m.append("a", 4)
    assert m.allocate("b", [1, 2, 3, 4, 5]) == 4       # [1,2] and [3,4] were filled by appends
    assert m.table("b")[:2] == [0, 1]


def test_model_no_blocks_changes_nothing():
    m = BlockManagerModel(2, 2)
    m.allocate("a", [1, 2, 3])
    free, ref = list(m.free), list(m.ref)
    assert not m.can_allocate([9, 9, 9])
    with pytest.raises(NoBlocks):
        m.allocate("b", [9, 9, 9])
    assert m.free == free and m.ref == ref and "b" not in m.seqs


# ------------------------------------------------------------------------------------------
# the library against the model
# ------------------------------------------------------------------------------------------

def _state_equal(bm, m, live):
    assert bm.num_free() == m.num_free()
    assert [bm.refcount(b) for b in range(m.N)] == m.ref
    for s in live:
        assert bm.block_table(s) == m.table(s), s
        assert bm.num_tokens(s) == len(m.seqs[s][0])


def _workload(seed, N, bs, ops, on_step, flags=0, model=True):
    """Seeded operations on the library (and on the model when `model`); on_step(kind, seq, x,
    got, got_model, bm, m, toks_of) checks each one. toks_of holds every live sequence's tokens
    as the library accepted them."""
    rng = np.random.default_rng(seed)
    systems = [list(rng.integers(0, 50, size=int(rng.integers(1, 4 * bs)))) for _ in range(4)]
    m = BlockManagerModel(N, bs) if model else None
    bm = pa.BlockManager(N, bs, flags)
    toks_of, next_id = {}, 0

    def admit(toks):
        nonlocal next_id
        got_m = None
        if m is not None:
            assert bm.can_allocate(toks) == m.can_allocate(toks)
            try:
                got_m = m.allocate(next_id, toks)
            except NoBlocks:
                pass
        try:
            got = bm.allocate(next_id, toks)
        except binding.BlockManagerError as e:
            assert e.code == -2
            got = None
        if got is not None:
            toks_of[next_id] = list(toks)
        on_step("allocate", next_id, toks, got, got_m, bm, m, toks_of)
        next_id += 1

    for _ in range(ops):
        r = rng.random()
        live = sorted(toks_of)
        if r < 0.35 or not live:
            sys_p = systems[int(rng.integers(0, len(systems)))]
            admit(sys_p + list(rng.integers(0, 50, size=int(rng.integers(1, 3 * bs)))))
        elif r < 0.85:
            s = live[int(rng.integers(0, len(live)))]
            t = int(rng.integers(0, 50))
            slot_m = None
            if m is not None:
                try:
                    slot_m = m.append(s, t)
                except NoBlocks:
                    pass
            try:
                slot = bm.append(s, t)
                toks_of[s].append(t)
            except binding.BlockManagerError as e:
                assert e.code == -2
                slot = None
            on_step("append", s, t, slot, slot_m, bm, m, toks_of)
        else:
            s = live[int(rng.integers(0, len(live)))]
            toks = toks_of.pop(s)
            if m is not None:
                m.release(s)
            bm.release(s)
            on_step("release", s, None, None, None, bm, m, toks_of)
            if r >= 0.95:                              # preemption: re-admitted with all its tokens
                admit(toks)
    return bm, m, toks_of


@pytest.mark.parametrize("seed,N,bs", [(0, 64, 4), (1, 40, 16), (2, 300, 1), (3, 24, 3),
                                       (4, 128, 8), (5, 16, 2)])
def test_library_matches_model(seed, N, bs):
    seen = {"hit": 0, "full": 0}

    def step(kind, s, x, got, got_m, bm, m, toks_of):
        assert got == got_m, (kind, s, got, got_m)
        _state_equal(bm, m, list(m.seqs))
        assert sorted(m.seqs) == sorted(toks_of)
        seen["hit"] += bool(kind == "allocate" and got)
        seen["full"] += got is None and kind != "release"
    _workload(seed, N, bs, 600, step)
    assert seen["hit"] > 0 and seen["full"] > 0   # the cache and the full pool were exercised


@pytest.mark.parametrize("seed,N,bs", [(10, 64, 4), (11, 40, 2), (12, 200, 1)])
def test_degenerate_hash_hits_stay_exact(seed, N, bs):
    """Every token hash equal: hits may be lost, never wrong. The test tracks what each block
    holds (the tokens from the sequence's start to the block's last written slot) from the
    library's own decisions."""
    content = {}
    hits = [0]

    def step(kind, s, x, got, got_m, bm, m, toks_of):
        if got is None or kind == "release":
            return
        toks = toks_of[s]
        table = bm.block_table(s)
        if kind == "allocate":
            assert got % bs == 0 and got < len(toks)
            hits[0] += got
            for i, b in enumerate(table):
                prefix = tuple(toks[:min((i + 1) * bs, len(toks))])
                if i < got // bs:
                    assert content.get(b) == prefix, "a hit on different content"
                else:
                    content[b] = prefix
        else:
            n = len(toks)
            b = table[(n - 1) // bs]
            assert got == b * bs + (n - 1) % bs
            content[b] = tuple(toks)

    bm, _, toks_of = _workload(seed, N, bs, 500, step, flags=pa.PA_BM_DEGENERATE_HASH, model=False)
    refs = [0] * N
    for q in toks_of:
        for b in bm.block_table(q):
            refs[b] += 1
    assert [bm.refcount(b) for b in range(N)] == refs
    assert bm.num_free() == sum(1 for r in refs if r == 0)


def test_library_errors():
    bm = pa.BlockManager(4, 2)
    assert bm.allocate(7, [1, 2, 3]) == 0
    with pytest.raises(binding.BlockManagerError) as e:
        bm.allocate(7, [1])
    assert e.value.code == -4
    with pytest.raises(binding.BlockManagerError) as e:
        bm.append(99, 1)
    assert e.value.code == -3
    with pytest.raises(binding.BlockManagerError) as e:
        bm.release(99)
    assert e.value.code == -3
    with pytest.raises(binding.BlockManagerError) as e:
        bm.allocate(8, [])
    assert e.value.code == -1
    free = bm.num_free()
    with pytest.raises(binding.BlockManagerError) as e:
        bm.allocate(8, [5, 5, 5, 5, 5])               # needs 3 blocks, 2 free
    assert e.value.code == -2 and bm.num_free() == free
    with pytest.raises(binding.BlockManagerError):
        bm.refcount(-1)
    with pytest.raises(binding.BlockManagerError):
        bm.refcount(4)
    with pytest.raises(binding.BlockManagerError):
        pa.BlockManager(0, 4)


def test_slots_feed_the_store():
    """The slots pa_bm_append returns are the pool rows pa_store_kv's slot_mapping addresses:
    block * block_size + offset, with the block from the sequence's table."""
    bm = pa.BlockManager(32, 4)
    bm.allocate(0, list(range(10)))
    for t in range(10, 30):
        slot = bm.append(0, t)
        table = bm.block_table(0)
        assert slot == table[t // 4] * 4 + t % 4
