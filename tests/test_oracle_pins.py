"""Pins of the oracle's building blocks against values it does not compute itself.

* SplitMix64: the published outputs of the generator started from 0, and an
  inverse derived here (un-xorshift, modular inverses of the multipliers).
* Held-out split (NeuronSpark-Trainer README, Concepts: 1 % of every file's
  documents by a hash of their text, 5 % for one source, the same in every
  line): the threshold's closed form, the hash's structure recovered through
  the inverse, order sensitivity, duplicate texts, seed independence and the
  binomial spread of the held-out count.
* Shuffle (same section: a file's documents are shuffled): the Feistel
  network inverted round by round, bijectivity of the cycle-walked
  permutation on every small domain, and its dependence on seed and stream.
"""
import math
import os
import random

import numpy as np
import pytest

import oracle
from _helpers import GOLDEN, corpus_from_lengths
from corpus import make_preset

M64 = (1 << 64) - 1
G = 0x9E3779B97F4A7C15
C1 = 0xBF58476D1CE4E5B9
C2 = 0x94D049BB133111EB


def _published_splitmix():
    out = []
    with open(os.path.join(GOLDEN, "splitmix64_seed0.txt")) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            n, v = line.split()
            out.append((int(n), int(v, 16)))
    return out


def _unxorshift(z, s):
    x = z
    for _ in range(64 // s + 1):
        x = z ^ (x >> s)
    return x


def _splitmix_inverse(y):
    z = _unxorshift(y, 31)
    z = (z * pow(C2, -1, 1 << 64)) & M64
    z = _unxorshift(z, 27)
    z = (z * pow(C1, -1, 1 << 64)) & M64
    z = _unxorshift(z, 30)
    return (z - G) & M64


# ---- SplitMix64 --------------------------------------------------------------
def test_splitmix64_published_outputs():
    for n, v in _published_splitmix():
        assert oracle.splitmix64(((n - 1) * G) & M64) == v


def test_splitmix64_inverts():
    rng = random.Random(5)
    for _ in range(2000):
        x = rng.getrandbits(64)
        assert _splitmix_inverse(oracle.splitmix64(x)) == x
    assert _splitmix_inverse(0xE220A8397B1DCDAF) == 0


# ---- held-out threshold ------------------------------------------------------
@pytest.mark.parametrize("bp", [1, 7, 100, 500, 5000, 9999])
def test_heldout_threshold_closed_form(bp):
    # floor(h * 10000 / 2^64) < bp  <=>  h < bp * 2^64 / 10000
    h0 = -(-(bp << 64) // 10000)  # ceil
    assert oracle.is_heldout(h0 - 1, bp)
    assert not oracle.is_heldout(h0, bp)
    assert oracle.is_heldout(0, bp)
    assert not oracle.is_heldout(M64, bp)


def test_heldout_rate_extremes():
    rng = random.Random(1)
    for _ in range(500):
        h = rng.getrandbits(64)
        assert not oracle.is_heldout(h, 0)
        assert oracle.is_heldout(h, 10000)
        # monotone in the rate
        flags = [oracle.is_heldout(h, bp) for bp in (0, 10, 100, 1000, 10000)]
        assert flags == sorted(flags)


# ---- the document hash -------------------------------------------------------
def test_doc_hash_empty_document_is_published_value():
    # with hash_key = -golden, the length term splitmix64(key + 0) is 0 and the
    # hash of an empty text is splitmix64(0): the first published output.
    assert oracle.doc_hash(np.zeros(0, np.int32), hash_key=(-G) & M64) == 0xE220A8397B1DCDAF


def test_doc_hash_structure_through_inverse():
    # With hash_key = -golden - L the length term vanishes, so the inverse of
    # the hash is the accumulated sum; growing a document by one token must add
    # exactly splitmix64((i << 32) | u32 token) to that sum.
    rng = np.random.default_rng(3)
    for L in (1, 2, 5, 33):
        toks = rng.integers(-2**31, 2**31, size=L, dtype=np.int64).astype(np.int32)
        prev = 0
        for k in range(1, L + 1):
            h = oracle.doc_hash(toks[:k], hash_key=(-G - k) & M64)
            acc = _splitmix_inverse(h)
            term = oracle.splitmix64(((k - 1) << 32) | (int(toks[k - 1]) & 0xFFFFFFFF))
            assert (acc - prev) & M64 == term
            prev = acc


def test_doc_hash_order_and_key_sensitivity():
    rng = np.random.default_rng(4)
    for _ in range(50):
        t = rng.integers(0, 50000, size=8).astype(np.int32)
        if t[0] == t[1]:
            continue
        s = t.copy()
        s[0], s[1] = t[1], t[0]
        assert oracle.doc_hash(t) != oracle.doc_hash(s)
        assert oracle.doc_hash(t, 0) != oracle.doc_hash(t, 1)
        assert oracle.doc_hash(t) != oracle.doc_hash(t[:-1])


def test_heldout_duplicate_text_same_decision_per_source():
    # Doc 0 is duplicated as doc 5 (same source) and doc 8 (another source);
    # the decision follows the text's hash and each source's own rate.
    rng = np.random.default_rng(9)
    lengths = [40, 30, 20, 25, 35, 40, 12, 14, 40, 22]
    toks = [rng.integers(0, 1000, size=L).astype(np.int32) for L in lengths]
    toks[5] = toks[0].copy()
    toks[8] = toks[0].copy()
    c = corpus_from_lengths(lengths, tokens=np.concatenate(toks), T=64, B=2, max_steps=1,
                            stream_docs=[6, 4], stream_source=[0, 1],
                            heldout_bp=[10000, 0])
    o = oracle.Oracle(c)
    flags, hashes = o.heldout()
    assert hashes[0] == hashes[5] == oracle.doc_hash(toks[0])
    assert flags[:6].all()          # rate 100 % in source 0
    assert not flags[6:].any()      # rate 0 in source 1
    # the same text in source 1 at a rate that keys on it
    for bp in (1, 100, 5000, 9999):
        c2 = corpus_from_lengths(lengths, tokens=np.concatenate(toks), T=64, B=2, max_steps=1,
                                 stream_docs=[6, 4], stream_source=[0, 1],
                                 heldout_bp=[bp, bp])
        f2, h2 = oracle.Oracle(c2).heldout()
        assert f2[0] == f2[5] == f2[8] == oracle.is_heldout(int(h2[0]), bp)


def test_heldout_rate_binomial_and_seed_independent():
    c = make_preset("c1")
    f0, _ = oracle.Oracle(c).heldout()
    f1, _ = oracle.Oracle(c, seed=12345).heldout()
    assert (f0 == f1).all()
    n, p = c.n_docs, 0.01
    mu, sd = n * p, math.sqrt(n * p * (1 - p))
    assert abs(int(f0.sum()) - mu) < 5 * sd


def test_heldout_rate_per_source_mixture():
    c = make_preset("c3s")
    f, _ = oracle.Oracle(c).heldout()
    sdb = c.stream_doc_begin
    for s in range(c.n_sources):
        js = [j for j in range(c.n_streams) if c.stream_source[j] == s]
        d0, d1 = int(sdb[js[0]]), int(sdb[js[-1] + 1])
        n = d1 - d0
        p = c.source_heldout_bp[s] / 10000.0
        mu, sd = n * p, math.sqrt(max(n * p * (1 - p), 1e-9))
        assert abs(int(f[d0:d1].sum()) - mu) <= 5 * sd + 1, (s, n, int(f[d0:d1].sum()))


# ---- the Feistel shuffle ------------------------------------------------------
@pytest.mark.parametrize("n,bits", [(0, 2), (1, 2), (2, 2), (4, 2), (5, 4), (16, 4), (17, 6),
                                    (1 << 20, 20), ((1 << 20) + 1, 22), ((1 << 31) + 5, 32)])
def test_feistel_domain_bits(n, bits):
    # max(2, ceil(log2 n)) rounded up to even
    assert oracle.feistel_bits(n) == bits


def _decrypt(keys, half, y):
    mask = (1 << half) - 1
    L, R = y >> half, y & mask
    for r in (3, 2, 1, 0):
        # a round maps (L, R) to (R, L ^ F_r(R)); undo it
        prevR = L
        prevL = R ^ (oracle.splitmix64(keys[r] ^ prevR) & mask)
        L, R = prevL, prevR
    return (L << half) | R


@pytest.mark.parametrize("half", [1, 2, 3, 5])
def test_feistel_rounds_invert_exhaustively(half):
    keys = [oracle.feistel_round_key(77, 3, r) for r in range(4)]
    dom = 1 << (2 * half)
    img = [oracle.feistel_encrypt(keys, half, x) for x in range(dom)]
    assert sorted(img) == list(range(dom))
    for x in range(dom):
        assert _decrypt(keys, half, img[x]) == x


def test_feistel_rounds_invert_wide():
    rng = random.Random(2)
    keys = [oracle.feistel_round_key(1, 0, r) for r in range(4)]
    fixed = 0
    for _ in range(3000):
        x = rng.getrandbits(32)
        y = oracle.feistel_encrypt(keys, 16, x)
        assert y < (1 << 32)
        assert _decrypt(keys, 16, y) == x
        fixed += (y == x)
    assert fixed <= 2


def test_feistel_pi_is_bijection_small_domains():
    for seed in (0, 1, 42, 2**63 + 5, 123456789):
        for n in list(range(1, 70)) + [97, 128, 129, 255, 256, 257, 300]:
            perm = [oracle.feistel_pi(seed, 2, n, p) for p in range(n)]
            assert sorted(perm) == list(range(n)), (seed, n)


def test_feistel_pi_is_first_in_range_point_of_orbit():
    n = 40  # domain 2^6 = 64: about a third of the points walk
    half = oracle.feistel_bits(n) // 2
    keys = [oracle.feistel_round_key(9, 1, r) for r in range(4)]
    walked = 0
    for p in range(n):
        y = oracle.feistel_encrypt(keys, half, p)
        steps = 1
        while y >= n:
            y = oracle.feistel_encrypt(keys, half, y)
            steps += 1
        walked += steps > 1
        assert oracle.feistel_pi(9, 1, n, p) == y
    assert walked > 0


def test_feistel_depends_on_seed_and_stream():
    n = 1000
    a = [oracle.feistel_pi(0, 0, n, p) for p in range(n)]
    b = [oracle.feistel_pi(1, 0, n, p) for p in range(n)]
    c = [oracle.feistel_pi(0, 1, n, p) for p in range(n)]
    assert a != b and a != c and b != c
    # a shuffled order, not a near-identity: few fixed points, low correlation
    assert sum(1 for p in range(n) if a[p] == p) < 10
    assert abs(np.corrcoef(np.arange(n), a)[0, 1]) < 0.15
