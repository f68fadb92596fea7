"""Pins for the CPU oracle: checks against facts fixed outside the oracle itself.

Each ``pin_*`` function takes an ``oracle.Oracle`` (the committed build, or a mutant build
made by ``test_oracle_mutants.py``) and raises ``AssertionError`` if the oracle disagrees with
what the pages and the mathematics fix:

* the 16-bit formats, against numpy's own float16 / float32 types;
* brute-force contiguous attention (``oracle.brute``) on tiny inputs whose pool was filled
  block by block with slice writes, not through the oracle's addressing;
* invariants the pages imply: output independent of block size (1, 4, 16, 256; "mini-vLLM"
  tests parity across block sizes) and of physical placement, batched equal to alone
  ("mini-vLLM": batched output against running alone), prefix-cached prefill equal to full
  recomputation (smzdm nano-vLLM deep dive: the prefix cache reuses already computed
  blocks; "nano-vLLM Part 4", section 3: prefill with an optional prefix block table);
* closed forms: one key gives its value, equal keys or a zero query give the mean value,
  designed scores give known softmax weights, per-head constant values expose the GQA map;
* the hand-derived fixture in ``tests/golden/closed_form_attention.json``.

Run as a script (``python tests/pins.py LIB``) it checks a given build and exits non-zero on
the first failing pin; the mutant tests use that to run each mutant in its own process.
"""
from __future__ import annotations

import json
import math
import sys
from pathlib import Path

import numpy as np

ROOT = Path(__file__).resolve().parents[1]
if str(ROOT) not in sys.path:
    sys.path.insert(0, str(ROOT))

from oracle import brute  # noqa: E402

GOLDEN = Path(__file__).resolve().parent / "golden"

TOL = 1e-12


def _rng(*seed):
    return np.random.default_rng(list(seed))


def _bits(x: np.ndarray, dtype: str) -> np.ndarray:
    """float64 -> storage bits (round to nearest even via numpy's float types)."""
    if dtype == "f16":
        return np.asarray(x, np.float64).astype(np.float16).view(np.uint16)
    f = np.asarray(x, np.float64).astype(np.float32).view(np.uint32)
    return ((f + (((f >> 16) & 1) + 0x7FFF)) >> 16).astype(np.uint16)


def _rand_bits(rng, shape, dtype):
    return _bits(rng.standard_normal(shape), dtype)


def _paged(seqs_k, seqs_v, block_size, rng=None, num_blocks=None, fill_bits=None):
    """Lay contiguous per-sequence rows [n_i, Hkv, D] into pools block by block.

    Physical IDs come from a permutation (identity without ``rng``); each sequence's b-th block
    receives rows b*bs .. b*bs+bs-1 by one slice assignment. Unused pool rows hold
    ``fill_bits`` (random if None), so a wrong address reads garbage, not zeros.
    """
    Hkv, D = seqs_k[0].shape[1:]
    nblk = [(k.shape[0] + block_size - 1) // block_size for k in seqs_k]
    total = sum(nblk)
    NB = num_blocks or max(total + 3, 1)
    ids = np.arange(NB) if rng is None else rng.permutation(NB)
    fill = _rng(99).integers(0, 0x3C00, size=(NB, block_size, Hkv, D), dtype=np.uint16) \
        if fill_bits is None else np.full((NB, block_size, Hkv, D), fill_bits, np.uint16)
    kc = fill.copy()
    vc = fill[::-1].copy()
    width = max(max(nblk), 1)
    bt = np.full((len(seqs_k), width), -1, np.int32)
    nxt = 0
    for i, (k, v) in enumerate(zip(seqs_k, seqs_v)):
        for b in range(nblk[i]):
            pid = int(ids[nxt])
            nxt += 1
            bt[i, b] = pid
            rows = slice(b * block_size, min((b + 1) * block_size, k.shape[0]))
            n = rows.stop - rows.start
            kc[pid, :n] = k[rows]
            vc[pid, :n] = v[rows]
    return kc, vc, bt


def _seqs(rng, lens, Hkv, D, dtype):
    ks = [_rand_bits(rng, (n, Hkv, D), dtype) for n in lens]
    vs = [_rand_bits(rng, (n, Hkv, D), dtype) for n in lens]
    return ks, vs


# ---------------------------------------------------------------------------------------------
# formats
# ---------------------------------------------------------------------------------------------

def pin_formats(orc):
    allbits = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    for dt in ("f16", "bf16"):
        mine = orc.bits_to_double(allbits, dt)
        ref = brute.bits_to_f64(allbits, dt)
        nan = np.isnan(ref)
        assert np.array_equal(np.isnan(mine), nan), dt
        assert np.array_equal(mine[~nan], ref[~nan]), dt
    # a few values by hand: 1.0, -2.0, the smallest fp16 subnormal, bf16 of 1.0
    assert orc.lib.oracle_f16_to_double(0x3C00) == 1.0
    assert orc.lib.oracle_f16_to_double(0xC000) == -2.0
    assert orc.lib.oracle_f16_to_double(0x0001) == 2.0 ** -24
    assert orc.lib.oracle_bf16_to_double(0x3F80) == 1.0


# ---------------------------------------------------------------------------------------------
# store
# ---------------------------------------------------------------------------------------------

def pin_store(orc):
    rng = _rng(1)
    NB, bs, Hkv, D = 7, 4, 2, 8
    T = 12
    canary = 0xA5A5
    kc = np.full((NB, bs, Hkv, D), canary, np.uint16)
    vc = np.full((NB, bs, Hkv, D), canary ^ 0xFFFF, np.uint16)
    k = rng.integers(0, 1 << 16, size=(T, Hkv, D), dtype=np.uint16)
    v = rng.integers(0, 1 << 16, size=(T, Hkv, D), dtype=np.uint16)
    slots = rng.choice(NB * bs, size=T, replace=False).astype(np.int32)
    slots[[2, 7]] = -1  # padding tokens
    k2, v2 = orc.store_kv(k, v, kc, vc, slots)
    fk = k2.reshape(NB * bs, Hkv, D)
    fv = v2.reshape(NB * bs, Hkv, D)
    written = set()
    for t, s in enumerate(slots):
        if s < 0:
            continue
        written.add(int(s))
        assert np.array_equal(fk[s], k[t]) and np.array_equal(fv[s], v[t]), t
    for s in range(NB * bs):
        if s not in written:
            assert (fk[s] == canary).all() and (fv[s] == (canary ^ 0xFFFF)).all(), s
    # contract violations are refused, not written
    for bad in ([0, 0], [NB * bs, 1]):
        try:
            orc.store_kv(k[:2], v[:2], kc, vc, np.array(bad, np.int32))
        except ValueError:
            pass
        else:
            raise AssertionError(f"slots {bad} accepted")


# ---------------------------------------------------------------------------------------------
# decode
# ---------------------------------------------------------------------------------------------

DECODE_SHAPES = [  # (B, Hq, Hkv, D, bs, dtype, lens)
    (3, 4, 2, 8, 4, "f16", [1, 5, 13]),
    (2, 6, 2, 16, 3, "bf16", [7, 20]),
    (3, 7, 1, 8, 16, "f16", [16, 17, 33]),
    (2, 8, 8, 4, 1, "bf16", [3, 6]),
]


def _decode_via_brute(q, ks, vs, scale, dt):
    out = []
    for i in range(len(ks)):
        qi = brute.bits_to_f64(q[i:i + 1], dt)
        out.append(brute.attention(qi, brute.bits_to_f64(ks[i], dt), brute.bits_to_f64(vs[i], dt),
                                   scale)[0])
    return np.stack(out)


def pin_decode_brute(orc):
    for n, (B, Hq, Hkv, D, bs, dt, lens) in enumerate(DECODE_SHAPES):
        rng = _rng(2, n)
        ks, vs = _seqs(rng, lens, Hkv, D, dt)
        q = _rand_bits(rng, (B, Hq, D), dt)
        kc, vc, bt = _paged(ks, vs, bs, rng)
        scale = 1.0 / math.sqrt(D)
        got = orc.decode(q, kc, vc, bt, np.array(lens, np.int32), scale=scale, dtype=dt)
        ref = _decode_via_brute(q, ks, vs, scale, dt)
        assert np.max(np.abs(got - ref)) <= TOL, (n, np.max(np.abs(got - ref)))


def pin_decode_block_size(orc):
    rng = _rng(3)
    lens = [1, 15, 16, 17, 300]
    Hq, Hkv, D, dt = 4, 2, 16, "bf16"
    ks, vs = _seqs(rng, lens, Hkv, D, dt)
    q = _rand_bits(rng, (len(lens), Hq, D), dt)
    outs = []
    for bs in (1, 4, 16, 256):
        kc, vc, bt = _paged(ks, vs, bs, _rng(3, bs))
        outs.append(orc.decode(q, kc, vc, bt, np.array(lens, np.int32), scale=0.25, dtype=dt))
    for o in outs[1:]:
        assert np.max(np.abs(o - outs[0])) <= TOL


def pin_decode_placement(orc):
    rng = _rng(4)
    lens = [9, 40, 2]
    Hq, Hkv, D, dt, bs = 6, 3, 8, "f16", 4
    ks, vs = _seqs(rng, lens, Hkv, D, dt)
    q = _rand_bits(rng, (3, Hq, D), dt)
    kc, vc, bt = _paged(ks, vs, bs, None)
    base = orc.decode(q, kc, vc, bt, np.array(lens, np.int32), scale=0.3, dtype=dt)
    perm = _rng(4, 1).permutation(kc.shape[0])          # physical block p moves to perm[p]
    kc2 = np.empty_like(kc)
    vc2 = np.empty_like(vc)
    kc2[perm] = kc
    vc2[perm] = vc
    bt2 = np.where(bt >= 0, perm[np.maximum(bt, 0)], -1).astype(np.int32)
    moved = orc.decode(q, kc2, vc2, bt2, np.array(lens, np.int32), scale=0.3, dtype=dt)
    assert np.array_equal(base, moved)


def pin_decode_batched_alone(orc):
    rng = _rng(5)
    lens = [5, 1, 23, 64]
    Hq, Hkv, D, dt, bs = 4, 1, 8, "bf16", 8
    ks, vs = _seqs(rng, lens, Hkv, D, dt)
    q = _rand_bits(rng, (4, Hq, D), dt)
    kc, vc, bt = _paged(ks, vs, bs, _rng(5, 1))
    batched = orc.decode(q, kc, vc, bt, np.array(lens, np.int32), scale=0.5, dtype=dt)
    for i in range(4):
        alone = orc.decode(q[i:i + 1], kc, vc, bt[i:i + 1], np.array(lens[i:i + 1], np.int32),
                           scale=0.5, dtype=dt)
        assert np.array_equal(alone[0], batched[i])


def pin_decode_closed_forms(orc):
    Hq, Hkv, D, bs, dt = 4, 2, 8, 4, "f16"
    G = Hq // Hkv
    rng = _rng(6)
    # (a) one key: the output is that key's value, exactly
    ks, vs = _seqs(rng, [1], Hkv, D, dt)
    q = _rand_bits(rng, (1, Hq, D), dt)
    kc, vc, bt = _paged(ks, vs, bs, rng)
    o = orc.decode(q, kc, vc, bt, np.array([1], np.int32), scale=0.7, dtype=dt)
    for h in range(Hq):
        assert np.array_equal(o[0, h], brute.bits_to_f64(vs[0][0, h // G], dt))
    # (b) all keys equal: uniform weights, the output is the mean of the values
    n = 11
    k_one = _rand_bits(rng, (1, Hkv, D), dt)
    ks = [np.repeat(k_one, n, axis=0)]
    vs = [_rand_bits(rng, (n, Hkv, D), dt)]
    kc, vc, bt = _paged(ks, vs, bs, rng)
    o = orc.decode(q, kc, vc, bt, np.array([n], np.int32), scale=0.7, dtype=dt)
    mean = brute.bits_to_f64(vs[0], dt).mean(axis=0)
    for h in range(Hq):
        assert np.max(np.abs(o[0, h] - mean[h // G])) <= TOL
    # (c) zero query: same
    ks, vs = _seqs(rng, [n], Hkv, D, dt)
    kc, vc, bt = _paged(ks, vs, bs, rng)
    qz = np.zeros((1, Hq, D), np.uint16)
    o = orc.decode(qz, kc, vc, bt, np.array([n], np.int32), scale=0.7, dtype=dt)
    mean = brute.bits_to_f64(vs[0], dt).mean(axis=0)
    for h in range(Hq):
        assert np.max(np.abs(o[0, h] - mean[h // G])) <= TOL
    # (d) GQA map: kv head g holds the constant value g + 1 in every row; q head h reads h//G + 1
    Hq2, Hkv2 = 6, 3
    ks, _ = _seqs(rng, [9], Hkv2, D, dt)
    vconst = np.zeros((9, Hkv2, D))
    for g in range(Hkv2):
        vconst[:, g, :] = g + 1
    vs = [_bits(vconst, dt)]
    kc, vc, bt = _paged(ks, vs, bs, rng)
    q6 = _rand_bits(rng, (1, Hq2, D), dt)
    o = orc.decode(q6, kc, vc, bt, np.array([9], np.int32), scale=0.7, dtype=dt)
    for h in range(Hq2):
        assert np.max(np.abs(o[0, h] - (h // (Hq2 // Hkv2) + 1))) <= TOL, h
    # (e) empty context: zero output
    o = orc.decode(q6, kc, vc, bt, np.array([0], np.int32), scale=0.7, dtype=dt)
    assert not o.any()


def pin_golden(orc):
    """Hand-derived fixture: scores chosen so the softmax weights are exact rationals."""
    fx = json.loads((GOLDEN / "closed_form_attention.json").read_text())
    for case in fx["cases"]:
        dt = case["dtype"]
        D = len(case["q"][0])
        keys = np.array(case["keys"], np.float64)[:, None, :]      # [n, 1, D]
        vals = np.array(case["values"], np.float64)[:, None, :]
        q = _bits(np.array(case["q"], np.float64)[None], dt)       # [1, 1, D]
        kc, vc, bt = _paged([_bits(keys, dt)], [_bits(vals, dt)], case["block_size"], _rng(7))
        o = orc.decode(q, kc, vc, bt, np.array([len(keys)], np.int32), scale=case["scale"],
                       dtype=dt)
        expect = np.array(case["expected_output"], np.float64)
        assert np.max(np.abs(o[0, 0] - expect)) <= 1e-12, (case["name"], o[0, 0], expect)


# ---------------------------------------------------------------------------------------------
# prefill
# ---------------------------------------------------------------------------------------------

def _prefill_inputs(rng, q_lens, P, Hq, Hkv, D, bs, dt):
    """Random full sequences (prefix + new rows); returns packed new rows and pools."""
    S = len(q_lens)
    kls = [P + ql for ql in q_lens]
    ks, vs = _seqs(rng, kls, Hkv, D, dt)
    q = _rand_bits(rng, (sum(q_lens), Hq, D), dt)
    cq = np.concatenate([[0], np.cumsum(q_lens)]).astype(np.int32)
    ck = np.concatenate([[0], np.cumsum(kls)]).astype(np.int32)
    kc, vc, bt = _paged(ks, vs, bs, rng)
    return S, ks, vs, q, cq, ck, kc, vc, bt


def pin_prefill_brute(orc):
    for n, (q_lens, P, Hq, Hkv, D, bs, dt, causal) in enumerate([
        ([5, 1, 9], 0, 4, 2, 8, 4, "f16", True),
        ([3, 7], 6, 6, 3, 8, 4, "bf16", True),
        ([4, 2], 5, 2, 1, 16, 3, "f16", False),
        ([1, 16, 17], 16, 8, 2, 4, 16, "bf16", True),
    ]):
        rng = _rng(8, n)
        S, ks, vs, q, cq, ck, kc, vc, bt = _prefill_inputs(rng, q_lens, P, Hq, Hkv, D, bs, dt)
        scale = 1.0 / math.sqrt(D)
        got_pool = orc.prefill(q, None, None, kc, vc, cq, ck, bt, Hkv=Hkv, block_size=bs,
                               scale=scale, dtype=dt, causal=causal)
        kp = np.concatenate(ks)
        vp = np.concatenate(vs)
        got_packed = orc.prefill(q, kp, vp, None, None, cq, ck, None, Hkv=Hkv, block_size=bs,
                                 scale=scale, dtype=dt, causal=causal)
        for s in range(S):
            qs = brute.bits_to_f64(q[cq[s]:cq[s + 1]], dt)
            ref = brute.attention(qs, brute.bits_to_f64(ks[s], dt), brute.bits_to_f64(vs[s], dt),
                                  scale, causal=causal)
            assert np.max(np.abs(got_pool[cq[s]:cq[s + 1]] - ref)) <= TOL, (n, s)
            assert np.max(np.abs(got_packed[cq[s]:cq[s + 1]] - ref)) <= TOL, (n, s)


def pin_prefill_prefix_recompute(orc):
    """Prefill of q new rows over a cached prefix of P rows equals the last q rows of a prefill
    of all P + q rows with nothing cached."""
    rng = _rng(9)
    q_lens, P, Hq, Hkv, D, bs, dt = [6, 1, 11], 8, 4, 2, 8, 4, "bf16"
    S, ks, vs, _, cq, ck, kc, vc, bt = _prefill_inputs(rng, q_lens, P, Hq, Hkv, D, bs, dt)
    full_q = [_rand_bits(rng, (P + ql, Hq, D), dt) for ql in q_lens]
    q_new = np.concatenate([fq[P:] for fq in full_q])
    cached = orc.prefill(q_new, None, None, kc, vc, cq, ck, bt, Hkv=Hkv, block_size=bs,
                         scale=0.4, dtype=dt)
    cf = ck.copy()
    full = orc.prefill(np.concatenate(full_q), np.concatenate(ks), np.concatenate(vs), None, None,
                       cf, cf, None, Hkv=Hkv, block_size=bs, scale=0.4, dtype=dt)
    for s in range(S):
        tail = full[cf[s] + P: cf[s + 1]]
        assert np.max(np.abs(cached[cq[s]:cq[s + 1]] - tail)) <= TOL, s


def pin_prefill_closed_forms(orc):
    """Zero queries: row r (position P + r) averages values 0..P+r; without causality, all."""
    rng = _rng(10)
    q_lens, P, Hq, Hkv, D, bs, dt = [4, 9], 5, 2, 1, 8, 4, "f16"
    S, ks, vs, _, cq, ck, kc, vc, bt = _prefill_inputs(rng, q_lens, P, Hq, Hkv, D, bs, dt)
    qz = np.zeros((sum(q_lens), Hq, D), np.uint16)
    for causal in (True, False):
        o = orc.prefill(qz, None, None, kc, vc, cq, ck, bt, Hkv=Hkv, block_size=bs, scale=1.0,
                        dtype=dt, causal=causal)
        for s in range(S):
            vals = brute.bits_to_f64(vs[s], dt)[:, 0]
            for r in range(q_lens[s]):
                n = P + r + 1 if causal else P + q_lens[s]
                for h in range(Hq):
                    assert np.max(np.abs(o[cq[s] + r, h] - vals[:n].mean(axis=0))) <= TOL
    # no prefix, causal: the first row of each prompt sees only itself
    o = orc.prefill(_rand_bits(rng, (sum(q_lens), Hq, D), dt),
                    np.concatenate([k[P:] for k in ks]), np.concatenate([v[P:] for v in vs]),
                    None, None, cq, cq, None, Hkv=Hkv, block_size=bs, scale=1.0, dtype=dt)
    for s in range(S):
        first = brute.bits_to_f64(vs[s][P], dt)[0]
        for h in range(Hq):
            assert np.array_equal(o[cq[s], h], first)


def pin_decode_is_last_prefill_row(orc):
    """A decode step over n cached tokens equals the last row of a causal prefill of n rows."""
    rng = _rng(11)
    lens, Hq, Hkv, D, bs, dt = [7, 19], 4, 2, 8, 4, "bf16"
    ks, vs = _seqs(rng, lens, Hkv, D, dt)
    kc, vc, bt = _paged(ks, vs, bs, rng)
    qfull = [_rand_bits(rng, (n, Hq, D), dt) for n in lens]
    cq = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    pre = orc.prefill(np.concatenate(qfull), None, None, kc, vc, cq, cq, bt, Hkv=Hkv,
                      block_size=bs, scale=0.3, dtype=dt)
    dec = orc.decode(np.stack([qf[-1] for qf in qfull]), kc, vc, bt, np.array(lens, np.int32),
                     scale=0.3, dtype=dt)
    for i in range(len(lens)):
        assert np.max(np.abs(dec[i] - pre[cq[i + 1] - 1])) <= TOL


ALL_PINS = [pin_formats, pin_store, pin_decode_brute, pin_decode_block_size, pin_decode_placement,
            pin_decode_batched_alone, pin_decode_closed_forms, pin_golden, pin_prefill_brute,
            pin_prefill_prefix_recompute, pin_prefill_closed_forms, pin_decode_is_last_prefill_row]


def main(argv):
    from oracle import Oracle
    orc = Oracle(argv[1]) if len(argv) > 1 else Oracle()
    for pin in ALL_PINS:
        try:
            pin(orc)
        except (AssertionError, ValueError) as e:
            print(f"FAIL {pin.__name__}: {e!r}")
            return 1
    print("all pins pass")
    return 0


if __name__ == "__main__":
    sys.exit(main(sys.argv))
