"""The attention split (host logic, no GPU): the (row, kv head, chunk) units a
decode launch cuts its attention into, through the library's own planning
query.  Pinned: the choices for the benchmarked workloads, the invariants the
kernel relies on (whole ring tiles per chunk, at most 64 chunks per row, the
partials buffer and the per-block unit bound), and that no other chunk has a
smaller estimated phase length under the documented cost."""
import random

import pytest

import synth
from synth import prompts as SP
from moe_decode_megakernel_persistent_gb300 import _lib as L

GRID = 152          # blocks of a launch on GB300 (one per SM)
TILE_INT4 = 30      # cached positions per ring tile, Flint int4 kernel
TILE_TINY = 60      # tiny-shape kernel (head_dim 64)


def _units(nkv, chunk, positions):
    return sum(nkv * ((p + 1 + chunk - 1) // chunk) for p in positions)


def _cost(units, chunk, tile, grid=GRID):
    return -(-units // grid) * (chunk + tile + tile // 2)


def _cap(nkv, grid=GRID):
    return min(4 * grid, grid + 16 * nkv)


@pytest.mark.parametrize("nkv,tile,positions,want", [
    (4, TILE_INT4, [2048], (60, 140)),          # batch 1, context 2049
    (4, TILE_INT4, [8022], (240, 136)),         # batch 1, context 8023
    (4, TILE_INT4, [2], (30, 4)),               # a short context: one tile per head
    (4, TILE_INT4, [2048] * 16, (1050, 128)),   # 16 rows at context 2049: one unit per block
    (2, TILE_TINY, [3000], (60, 102)),          # the tiny shape's long-context test
])
def test_plan_for_the_benchmarked_workloads(nkv, tile, positions, want):
    assert L.mk_attention_plan(nkv, GRID, tile, positions) == want


def test_the_16_client_workload_takes_one_unit_per_block():
    lengths = [n for _, n in SP.schedule(synth.CONFIGS[5])]
    chunk, units = L.mk_attention_plan(4, GRID, TILE_INT4, lengths)
    assert units == GRID
    assert units == _units(4, chunk, lengths)


def test_plan_invariants_and_optimality_on_random_batches():
    rng = random.Random(8)
    for _ in range(120):
        nkv = rng.choice([1, 2, 4, 8])
        tile = rng.choice([16, 30, 60])
        grid = rng.choice([1, 7, 152])
        positions = [rng.randrange(0, rng.choice([40, 2000, 9000])) for _ in range(rng.randrange(1, 17))]
        chunk, units = L.mk_attention_plan(nkv, grid, tile, positions)
        longest = max(positions) + 1
        assert chunk % tile == 0 and chunk >= tile
        assert units == _units(nkv, chunk, positions)
        assert -(-longest // chunk) <= 64
        cap = _cap(nkv, grid)
        if units > cap:  # only the one-chunk-per-row fallback may exceed the bound
            assert units == nkv * len(positions)
            continue
        best = _cost(units, chunk, tile, grid)
        c = tile
        while True:  # no other whole-tile chunk within the bounds is estimated shorter
            u = _units(nkv, c, positions)
            if u <= cap and -(-longest // c) <= 64:
                cost = _cost(u, c, tile, grid)
                assert cost >= best, (nkv, grid, tile, positions, chunk, c)
                if cost == best:
                    assert c <= chunk  # ties go to the larger chunk
            if c >= longest:
                break
            c += tile


def test_plan_rejects_bad_arguments():
    for args in ((0, GRID, TILE_INT4, [5]), (4, 0, TILE_INT4, [5]), (4, GRID, 0, [5]),
                 (4, GRID, TILE_INT4, [-1]), (4, GRID, TILE_INT4, [5] * 17)):
        with pytest.raises(L.MKError) as e:
            L.mk_attention_plan(*args)
        assert e.value.code == L.MK_ERR_INVALID_ARG
