"""The bench's algorithmic-work formulas, pinned by brute force (CPU).

Every roofline fraction the bench reports divides a FLOP or byte count by a
measured time; these counts must be the work the definition implies (only
visible (row, key) pairs, each request's keys read once), not what a kernel
happens to execute.  Counts are taken here row by row from the oracle's own
visibility rule.
"""

import numpy as np
import pytest

import bench
from oracle.paged_attention import first_visible_key, row_position, visible_keys

HEADS = (32, 8, 128)
CASES = [([1], [1]), ([3], [64]), ([64], [64]), ([5, 0, 17, 1], [9, 4, 17, 300]), ([128, 7], [4096, 4103])]


def brute_pairs(q_lens, kv_lens, window=0):
    total = 0
    for q, kv in zip(q_lens, kv_lens):
        for i in range(q):
            p = row_position(i, q, kv)
            total += visible_keys(p) - first_visible_key(p, window)
    return total


def brute_keys(q_lens, kv_lens, window=0):
    total = 0
    for q, kv in zip(q_lens, kv_lens):
        seen = np.zeros(kv, dtype=bool)
        for i in range(q):
            p = row_position(i, q, kv)
            seen[first_visible_key(p, window):visible_keys(p)] = True
        total += int(seen.sum())
    return total


@pytest.mark.parametrize("q_lens,kv_lens", CASES)
def test_flops_count_visible_pairs_only(q_lens, kv_lens):
    hq, _, d = HEADS
    assert bench.flops_of(HEADS, q_lens, kv_lens) == 4 * d * hq * brute_pairs(q_lens, kv_lens)
    for q, kv in zip(q_lens, kv_lens):
        assert bench.pairs(q, kv) == brute_pairs([q], [kv])


@pytest.mark.parametrize("q_lens,kv_lens", CASES)
def test_kv_bytes_read_every_key_once(q_lens, kv_lens):
    # a causal row set reads keys 0 .. kv_len - 1 (the last row sees them all), K and V
    _, hkv, d = HEADS
    for elem in (2, 1):
        assert bench.kv_bytes_of(HEADS, kv_lens, elem) == sum(kv * 2 * hkv * d * elem for kv in kv_lens)
    assert all(brute_keys([q], [kv]) == (kv if q else 0) for q, kv in zip(q_lens, kv_lens))


@pytest.mark.parametrize("window", [1, 16, 100, 4096])
@pytest.mark.parametrize("q_lens,kv_lens", CASES)
def test_windowed_work_matches_the_window_definition(q_lens, kv_lens, window):
    hq, hkv, d = HEADS
    fl, kvb = bench.windowed_work(HEADS, q_lens, kv_lens, window)
    assert fl == 4 * d * hq * brute_pairs(q_lens, kv_lens, window)
    # keys read: the union of the rows' windows (requests with no rows read none)
    assert kvb == brute_keys(q_lens, kv_lens, window) * 2 * hkv * d * 2


def test_window_at_least_the_sequence_is_plain_causal():
    q_lens, kv_lens = [5, 17, 128], [9, 17, 4103]
    fl, _ = bench.windowed_work(HEADS, q_lens, kv_lens, 5000)
    assert fl == bench.flops_of(HEADS, q_lens, kv_lens)


@pytest.mark.parametrize("kind", ["half", "documents"])
def test_profile_mask_density_and_shape(kind):
    # the profile's packed mask, unpacked: its reported density is the visible
    # share of causal pairs; a document mask shows each row a contiguous run of
    # keys that ends at the row's own position
    b = bench.make_batch((8, 2, 128), 3, 700, 5000, "cpu")
    words, density = bench.profile_mask(b, kind, seed=1)
    assert words.dtype == np.int32 and words.shape == (b.total_q, (5000 + 31) // 32)
    bits = np.unpackbits(words.view(np.uint8), axis=1, bitorder="little").astype(bool)
    visible = causal = 0
    for r in range(b.batch):
        lo, hi = b.row_range(r)
        ql, kl = b.q_lens[r], b.kv_lens[r]
        for i in range(ql):
            p = row_position(i, ql, kl)
            seen = bits[lo + i, :p + 1]
            visible += int(seen.sum())
            causal += p + 1
            if kind == "documents":
                first = int(np.argmax(seen))
                assert seen[p] and seen[first:].all() and not seen[:first].any()
                assert p - first < 4096
    assert abs(density - visible / causal) < 1e-12
    assert (0.45 < density < 0.55) if kind == "half" else (0.0 < density < 0.5)
