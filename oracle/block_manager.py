"""Reference model of the host block manager: the plain statement, no performance concerns.

TEST INFRASTRUCTURE (see the package docstring): only tests and bench.py's CPU leg use it.

What it models (nano-vLLM Part 4, sections 2 and 3: block IDs, reference counts and prefix-hash
metadata, "exact full-block prefix cache", free on finish; smzdm deep dive "调度与内存": blocks of
256 tokens, reference counts, a prefix cache that lets sequences sharing a system prompt reuse
blocks, preemption that frees blocks but keeps the tokens; mini-vLLM: a preallocated pool, an O(1)
free-list allocator, a block table per sequence). Where the pages stop, the readings are:

* The pool holds blocks 0 .. N-1 of `block_size` token slots. Free blocks wait in a first-in
  first-out queue, initially in id order; a block whose last reference goes away joins the back.
* A full block is identified by its parent (the block before it in the sequence that filled it,
  or the root) and its own tokens. Because a block taken from the free queue for new content gets a
  new identity (its old cached content is forgotten, and so are the blocks cached after it), a
  match on (parent, tokens) is a match on the whole prefix: the cache is exact. Here the key is the
  parent's identity and the tuple of tokens, with no hash at all.
* A new sequence reuses the longest run of cached full blocks from its start, except a block that
  would hold its last token: at least one token is always computed. Reused blocks gain a
  reference (a reused block that was free leaves the free queue); the other blocks come from the
  front of the free queue. Full blocks among them are cached at once (their tokens are known).
* Appending a token takes a new block from the free queue when the last block is full; a block
  that becomes full is cached.
* Freeing a sequence drops one reference from each of its blocks, last block first; blocks left
  with none join the back of the free queue and stay findable until they are taken for new content.
* The most recently cached block wins when two blocks hold the same (parent, tokens).
"""
from __future__ import annotations

ROOT = -1


class NoBlocks(Exception):
    pass


class BlockManagerModel:
    def __init__(self, num_blocks: int, block_size: int):
        assert num_blocks >= 1 and block_size >= 1
        self.N, self.bs = num_blocks, block_size
        self.free = list(range(num_blocks))   # front = index 0
        self.ref = [0] * num_blocks
        self.gen = [0] * num_blocks           # identity of the block's current content
        self.key = [None] * num_blocks        # (parent identity, tokens) while cached
        self.cache: dict = {}                 # (parent identity, tokens) -> block
        self.seqs: dict = {}                  # seq -> (tokens list, table list)

    def node(self, b: int):
        return ROOT if b == ROOT else (b, self.gen[b])

    def _take_free(self) -> int:
        b = self.free.pop(0)
        k = self.key[b]
        if k is not None and self.cache.get(k) == b:
            del self.cache[k]
        self.key[b] = None
        self.gen[b] += 1                      # new content: a new identity
        return b

    def _cache(self, b: int, parent: int, toks):
        k = (self.node(parent), tuple(toks))
        self.key[b] = k
        self.cache[k] = b

    def _match(self, tokens):
        n, bs = len(tokens), self.bs
        matched, parent = [], ROOT
        for i in range((n - 1) // bs):         # blocks that end before the last token
            b = self.cache.get((self.node(parent), tuple(tokens[i * bs:(i + 1) * bs])))
            if b is None:
                break
            matched.append(b)
            parent = b
        return matched

    def can_allocate(self, tokens) -> bool:
        matched = self._match(tokens)
        total = -(-len(tokens) // self.bs)
        need = total - len(matched) + sum(1 for b in matched if self.ref[b] == 0)
        return need <= len(self.free)

    def allocate(self, seq, tokens) -> int:
        """Blocks for a new sequence; returns the number of its tokens already cached."""
        tokens = list(tokens)
        assert len(tokens) >= 1 and seq not in self.seqs
        if not self.can_allocate(tokens):
            raise NoBlocks
        bs = self.bs
        matched = self._match(tokens)
        for b in matched:
            if self.ref[b] == 0:
                self.free.remove(b)
            self.ref[b] += 1
        table = list(matched)
        parent = matched[-1] if matched else ROOT
        total = -(-len(tokens) // bs)
        for i in range(len(matched), total):
            b = self._take_free()
            self.ref[b] = 1
            if (i + 1) * bs <= len(tokens):    # a full block: cached now
                self._cache(b, parent, tokens[i * bs:(i + 1) * bs])
            table.append(b)
            parent = b
        self.seqs[seq] = (tokens, table)
        return len(matched) * bs

    def append(self, seq, token) -> int:
        """One more token; returns its slot."""
        tokens, table = self.seqs[seq]
        bs, n = self.bs, len(tokens)
        if n % bs == 0:
            if not self.free:
                raise NoBlocks
            b = self._take_free()
            self.ref[b] = 1
            table.append(b)
        tokens.append(token)
        blk = table[n // bs]
        if (n + 1) % bs == 0:
            i = n // bs
            self._cache(blk, table[i - 1] if i > 0 else ROOT, tokens[i * bs:(i + 1) * bs])
        return blk * bs + n % bs

    def release(self, seq):
        tokens, table = self.seqs.pop(seq)
        for b in reversed(table):
            self.ref[b] -= 1
            if self.ref[b] == 0:
                self.free.append(b)

    def table(self, seq):
        return list(self.seqs[seq][1])

    def num_free(self) -> int:
        return len(self.free)
