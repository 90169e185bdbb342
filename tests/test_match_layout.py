"""Host restatement of the Match kernels' data layout (no GPU): which ring
entry and column every 16-byte load of a lane holds, the transposing
half-warp reduction that leaves each lane one entry's distance, and how a
query group is split over Match blocks.  A mistake in any of these index
maps would pair a lane with the wrong entry; here each is checked against a
direct sum, entry by entry."""
import numpy as np
import pytest

LANES, CHUNKS_PER_ENTRY = 32, 16   # 128 bf16 = 16 chunks of 16 bytes


def lane_loads(partial, ring_len, n_loads):
    """v[lane][i]: the partial distance lane `lane` forms from load i, which
    is chunk 32 i + lane of the head's [L][16] block (zero past the ring)."""
    v = np.zeros((LANES, 16))
    for lane in range(LANES):
        for i in range(n_loads):
            ch = 32 * i + lane
            e, col = divmod(ch, CHUNKS_PER_ENTRY)
            assert e == 2 * i + (lane >> 4) and col == lane & 15
            if ch < ring_len * CHUNKS_PER_ENTRY:
                v[lane, i] = partial[e, col]
    return v


def halve_sum(v, n):
    """One step for n values per lane: lane bit n/2 picks the half it keeps
    and it adds its partner's copy of that half."""
    o = n // 2
    out = v.copy()
    for lane in range(LANES):
        up = bool(lane & o)
        partner = lane ^ o
        pup = bool(partner & o)
        for k in range(o):
            keep = v[lane, k + o] if up else v[lane, k]
            recv = v[partner, k] if pup else v[partner, k + o]
            out[lane, k] = keep + recv
    return out


@pytest.mark.parametrize("ring_len,n_loads", [(1, 8), (5, 8), (16, 8), (17, 16), (31, 16), (32, 16)])
def test_each_lane_ends_with_its_entrys_distance(ring_len, n_loads):
    rng = np.random.default_rng(ring_len)
    partial = rng.random((32, CHUNKS_PER_ENTRY))   # per (entry, column) squared-difference sums
    v = lane_loads(partial, ring_len, n_loads)
    for n in (16, 8, 4, 2):
        v = halve_sum(v, n)
    owners = {}
    for lane in range(LANES):
        e = 2 * (lane & 15) + (lane >> 4)
        owners.setdefault(e, []).append(lane)
        if e < ring_len:
            assert v[lane, 0] == pytest.approx(partial[e].sum(), rel=1e-12)
    assert sorted(owners) == list(range(32)) and all(len(x) == 1 for x in owners.values())


def test_eight_loads_cover_sixteen_entries_and_sixteen_cover_thirty_two():
    for n_loads, entries in ((8, 16), (16, 32)):
        seen = {divmod(32 * i + lane, CHUNKS_PER_ENTRY) for i in range(n_loads) for lane in range(LANES)}
        assert seen == {(e, c) for e in range(entries) for c in range(CHUNKS_PER_ENTRY)}


@pytest.mark.parametrize("G", [1, 2, 4, 8, 16, 32])
def test_group_split_over_match_blocks_covers_every_head_once(G):
    parts = (G + 7) // 8             # at most 8 heads (warps) per block
    nw = (G + parts - 1) // parts
    heads = [part * nw + w for part in range(parts) for w in range(nw) if part * nw + w < G]
    assert sorted(heads) == list(range(G)) and nw <= 8
