"""Pins for the oracle's packed key, slot hash and sequential linear-probing
table ("What Irregularity Costs", design section: 16-byte entries with a
64-bit key packing the three block coordinates, each biased by 2^20 into 21
bits; open addressing with linear probing; a multiply-xor hash).

The pins come from outside the oracle:
* the key layout's special values, derived by hand from the bit layout;
* round trips over every boundary combination and random coordinates;
* two theorems about linear probing with insertions only: the set of
  occupied slots and the total displacement do not depend on the insertion
  order (Peterson 1957; Knuth, TAOCP vol. 3, 6.4) -- the same property the
  GPU table is checked against;
* Knuth's expected successful-search cost for random keys,
  (1 + 1 / (1 - alpha)) / 2;
* a brute-force Python linear-probing table on tiny sizes, including
  wrap-around at the end of the table.
"""
import random

import numpy as np
import pytest

B20 = 1 << 20


def test_key_special_values(oracle_mod):
    # all three fields at their minimum: every biased field is 0
    assert oracle_mod.pack_key(-B20, -B20, -B20) == 0
    # all three at their maximum: 63 one bits, bit 63 clear
    assert oracle_mod.pack_key(B20 - 1, B20 - 1, B20 - 1) == (1 << 63) - 1
    # the origin: each field holds 2^20
    assert oracle_mod.pack_key(0, 0, 0) == (1 << 20) | (1 << 41) | (1 << 62)
    # one field at a time: x occupies bits 0-20, y bits 21-41, z bits 42-62
    assert oracle_mod.pack_key(5, -B20, -B20) == 5 + B20
    assert oracle_mod.pack_key(-B20, 5, -B20) == (5 + B20) << 21
    assert oracle_mod.pack_key(-B20, -B20, 5) == (5 + B20) << 42
    assert oracle_mod.pack_key(-1, -B20, -B20) == B20 - 1


def test_key_roundtrip_boundaries(oracle_mod):
    edge = [-B20, -B20 + 1, -2, -1, 0, 1, 2, B20 - 2, B20 - 1]
    seen = set()
    for x in edge:
        for y in edge:
            for z in edge:
                k = oracle_mod.pack_key(x, y, z)
                assert k is not None and k >> 63 == 0
                assert oracle_mod.unpack_key(k) == (x, y, z)
                seen.add(k)
    assert len(seen) == len(edge) ** 3


def test_key_roundtrip_random(oracle_mod):
    rng = np.random.Generator(np.random.PCG64(11))
    c = rng.integers(-B20, B20, size=(100_000, 3))
    keys = oracle_mod.pack_keys(c)
    assert np.unique(keys).size == np.unique(c, axis=0).shape[0]
    for i in range(0, c.shape[0], 997):
        assert oracle_mod.unpack_key(int(keys[i])) == tuple(int(v) for v in c[i])


@pytest.mark.parametrize("bad", [(-B20 - 1, 0, 0), (0, B20, 0), (0, 0, B20), (0, 0, -(1 << 31))])
def test_key_rejects_out_of_range(oracle_mod, bad):
    assert oracle_mod.pack_key(*bad) is None


def test_unpack_rejects_empty_marker(oracle_mod):
    assert oracle_mod.unpack_key((1 << 64) - 1) is None


def test_hash_slots_in_range_and_spread(oracle_mod):
    # a dense cube of neighbouring blocks (the typical key pattern) spreads
    # over a 2^12 table like a uniform draw: chi-square within 5 sigma
    T = 1 << 12
    counts = np.zeros(T, dtype=np.int64)
    n = 0
    for x in range(-8, 24):
        for y in range(-8, 24):
            for z in range(-8, 24):
                s = oracle_mod.hash_slot(oracle_mod.pack_key(x, y, z), T)
                assert 0 <= s < T
                counts[s] += 1
                n += 1
    expected = n / T
    chi2 = float(((counts - expected) ** 2 / expected).sum())
    assert abs(chi2 - (T - 1)) < 5 * np.sqrt(2 * (T - 1))


def test_hash_slots_of_large_tables_distinct(oracle_mod):
    # slots in a 2^62-slot table keep 62 bits of a bijective 64-bit mix, so
    # 20,000 distinct keys must land in 20,000 distinct slots
    rng = np.random.Generator(np.random.PCG64(5))
    c = np.unique(rng.integers(-B20, B20, size=(20_000, 3)), axis=0)
    keys = oracle_mod.pack_keys(c)
    slots = {oracle_mod.hash_slot(int(k), 1 << 62) for k in keys}
    assert len(slots) == len(keys)


def _python_linear_probe(keys, T, home):
    table = [None] * T
    lens = []
    for k in keys:
        s = home[k]
        n = 1
        while table[s] is not None and table[s] != k:
            s = (s + 1) % T
            n += 1
        if table[s] is None:
            table[s] = k
        lens.append(n)
    return table, lens


def test_probe_build_matches_bruteforce_with_wraparound(oracle_mod):
    T = 64
    # keys whose home slots sit at the end of the table, so chains wrap to 0
    coords = oracle_mod.clustered_coords(T, T - 4, 4, (-30, 7, 2), 40, 20)
    assert coords.shape[0] == 20
    keys = [int(k) for k in oracle_mod.pack_keys(coords)]
    keys = keys + keys[:5]                       # repeats are found, not re-inserted
    home = {k: oracle_mod.hash_slot(k, T) for k in keys}
    assert all(T - 4 <= home[k] < T for k in keys)
    table, lens, disp, distinct = oracle_mod.probe_build(np.array(keys, dtype=np.uint64), T)
    ref_table, ref_lens = _python_linear_probe(keys, T, home)
    empty = np.uint64((1 << 64) - 1)
    assert [None if t == empty else int(t) for t in table] == ref_table
    assert list(lens) == ref_lens
    assert distinct == 20
    # 20 keys homed in the last 4 slots fill slots 60..63 and wrap to 0..15
    occupied = sorted(i for i, t in enumerate(ref_table) if t is not None)
    assert occupied == list(range(0, 16)) + list(range(60, 64))


def test_probe_build_order_invariance(oracle_mod):
    rng = random.Random(7)
    T = 1 << 12
    c = np.unique(np.random.Generator(np.random.PCG64(3)).integers(-500, 500, size=(1800, 3)),
                  axis=0)
    keys = [int(k) for k in oracle_mod.pack_keys(c)]
    ref_table, _, ref_disp, _ = oracle_mod.probe_build(np.array(keys, dtype=np.uint64), T)
    empty = np.uint64((1 << 64) - 1)
    ref_occ = ref_table != empty
    for _ in range(5):
        rng.shuffle(keys)
        table, _, disp, distinct = oracle_mod.probe_build(np.array(keys, dtype=np.uint64), T)
        assert distinct == len(keys)
        assert np.array_equal(table != empty, ref_occ)
        assert disp == ref_disp


@pytest.mark.parametrize("alpha", [0.1, 0.3, 0.5])
def test_probe_mean_matches_knuth(oracle_mod, alpha):
    T = 1 << 16
    n = int(alpha * T)
    c = np.unique(np.random.Generator(np.random.PCG64(17)).integers(-B20, B20, size=(n, 3)),
                  axis=0)
    keys = oracle_mod.pack_keys(c)
    _, _, disp, distinct = oracle_mod.probe_build(keys, T)
    mean_success = 1.0 + disp / distinct
    a = distinct / T
    knuth = 0.5 * (1.0 + 1.0 / (1.0 - a))
    assert abs(mean_success - knuth) / knuth < 0.05


def test_clustered_coords_form_one_long_chain(oracle_mod):
    T = 1 << 12
    w = T // 64
    want = T // 2
    coords = oracle_mod.clustered_coords(T, 1000, w, (0, 0, 0), 64, want)
    assert coords.shape[0] == want
    keys = oracle_mod.pack_keys(coords)
    assert all(1000 <= oracle_mod.hash_slot(int(k), T) < 1000 + w for k in keys[:200])
    table, plen, disp, distinct = oracle_mod.probe_build(keys, T)
    # the keys fill one run of `want` consecutive slots starting at the window
    occ = np.nonzero(table != np.uint64((1 << 64) - 1))[0]
    assert np.array_equal(occ, np.arange(1000, 1000 + want))
    # mean displacement is about half the run length
    assert disp / distinct > want / 2 - w


def test_hash_known_answers_from_the_published_splitmix64_sequence(oracle_mod):
    """The slot hash is the SplitMix64 output mix: on the states that give
    the generator's published outputs it must return those outputs (here
    to 63 bits, the largest power-of-two table the call accepts, and masked
    to the table sizes of the workloads)."""
    import helpers
    vectors = helpers.splitmix64_vectors()
    assert len(vectors) == 5
    for state, value in vectors:
        assert oracle_mod.hash_slot(state, 1 << 63) == value % (1 << 63)
        for T in (1 << 14, 1 << 16, 1 << 18, 1 << 21):
            assert oracle_mod.hash_slot(state, T) == value % T


@pytest.mark.parametrize("mutant,what", [(23, "last xor-shift by 32 instead of 31"),
                                         (24, "first multiplier used for the second")])
def test_hash_mistakes_pass_the_spread_pins_but_not_the_known_answers(oracle_mod, mutant, what):
    """A wrong shift or constant still spreads keys well (the structural
    pins cannot see it); the published outputs reject it."""
    import os

    import helpers
    try:
        vectors = helpers.splitmix64_vectors()
        wrong = [s for s, v in vectors
                 if oracle_mod.hash_slot(s, 1 << 63, mutant=mutant) != v % (1 << 63)]
        assert wrong, f"the known-answer pin misses the planted mistake: {what}"
    finally:
        path = oracle_mod.library_path(mutant)
        if os.path.exists(path):
            os.remove(path)
