"""Invariants of the GEMM's split of a fractional wave over the CTA pairs
(host model in split_tail_ref, which restates the kernel's assignment): every
K block of every tile is computed exactly once; a split tile has exactly one
head and one tail, on consecutive units; every unit's head is its first item,
so a tail never waits on a unit that is itself waiting; the split work comes
before the whole tiles; the units' shares differ by at most one tile."""
import itertools

import pytest

from split_tail_ref import plan_split, work_items, tile_rows


@pytest.mark.parametrize("T,units,num_kb", list(itertools.product(
    (1, 5, 75, 76, 77, 80, 110, 151, 152, 153, 200, 648, 864, 1000),
    (1, 2, 3, 76, 148),
    (1, 2, 7, 20, 48, 192))))
def test_every_block_once_and_one_handover_per_split_tile(T, units, num_kb):
    units = min(units, T)
    sk = plan_split(T, units)
    if sk:
        assert units < sk < 2 * units and (T - sk) % units == 0
    cover = {}
    heads, tails = {}, {}
    work = []
    for u in range(units):
        items = work_items(u, units, T, sk, num_kb)
        work.append(sum(kb1 - kb0 for _, kb0, kb1, _ in items))
        kinds = [k for _, _, _, k in items]
        assert kinds.count("head") <= 1 and kinds.count("tail") <= 1
        if "head" in kinds:
            assert kinds.index("head") == 0
        n_split = sum(1 for t, *_ in items if t < sk)
        assert all(t < sk for t, *_ in items[:n_split])        # split items first
        if "tail" in kinds:
            assert kinds.index("tail") == n_split - 1            # the last split item
        for t, kb0, kb1, kind in items:
            assert 0 <= kb0 < kb1 <= num_kb
            if kind == "head":
                assert kb0 == 0 and kb1 < num_kb and t < sk
                heads[t] = u
            if kind == "tail":
                assert kb0 > 0 and kb1 == num_kb and t < sk
                tails[t] = u
            for kb in range(kb0, kb1):
                assert (t, kb) not in cover
                cover[(t, kb)] = u
    assert len(cover) == T * num_kb
    assert set(heads) == set(tails)
    for t in heads:
        assert tails[t] == heads[t] + 1
    if sk:
        assert max(work) - min(work) <= 1


def test_split_only_where_it_pays():
    assert plan_split(648, 76) == 116          # DiT QKV: 8.53 waves of 256 x 256 tiles
    assert plan_split(612, 76) == 80           # 8.05 waves
    assert plan_split(684, 76) == 0            # 9 full waves
    assert plan_split(216, 76) == 0            # 2.84 waves: the last wave is busy enough
    assert plan_split(46 + 76 * 3, 76) == 0    # 30 of 76 idle: under 40 %
    assert plan_split(45 + 76 * 3, 76) == 76 + 45  # 31 of 76 idle
    assert plan_split(108, 76) == 0            # no whole wave would remain
    assert plan_split(40, 76) == 0


def test_tile_height_choice():
    # with the split, 256-row tiles win on the large shapes
    assert tile_rows(4608, [3072] * 3, 76, True) == 256
    assert tile_rows(4352, [3072] * 3, 76, True) == 256
    assert tile_rows(4608, [12288], 76, True) == 256
    # under two waves no split: two waves of 192-row tiles beat 256-row ones
    assert tile_rows(768, [3072] * 3, 76, True) == 192
    assert tile_rows(4096, [1280], 76, True) == 192   # only 256-row tiles split
    # one wave either way: the shortest tile gives the most parallelism
    assert tile_rows(256, [3072], 76, True) == 128
