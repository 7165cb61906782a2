"""Host model of how the GEMM shares its output tiles among its CTA pairs
("units"), used by the tests to state the split's invariants and to pick
shapes that exercise it.

When a last wave of whole tiles would leave at least 40 % of the units idle
and at least one whole wave remains, the first (fractional wave + one whole
wave) tiles are split: their K
blocks, laid out tile after tile, are cut into one contiguous range per unit,
and every unit does its range first. A unit whose range ends inside a tile
(the tile's head) hands its int32 partial sums to the unit whose range
finishes the tile (the tail), which is always the next unit. The remaining
tiles are then taken whole, round-robin over the units.
"""


def split_pays(T: int, units: int) -> bool:
    if units < 2 or T < 2 * units:
        return False
    rem = T % units
    return rem != 0 and 10 * (units - rem) >= 4 * units


def plan_split(total_tiles: int, units: int) -> int:
    """Number of split tiles (at the start of the tile order) for `units` units."""
    if not split_pays(total_tiles, units):
        return 0
    return units + total_tiles % units


def work_items(unit: int, units: int, total_tiles: int, sk: int, num_kb: int):
    """The unit's items in its order: (tile, kb0, kb1, kind), kind in
    {"whole", "head", "tail"}."""
    items = []
    if sk:
        total = sk * num_kb
        s, e = total * unit // units, total * (unit + 1) // units
        for tile in range((e - 1) // num_kb, s // num_kb - 1, -1):
            base = tile * num_kb
            kb0, kb1 = max(0, s - base), min(num_kb, e - base)
            kind = "head" if kb1 < num_kb else ("tail" if kb0 > 0 else "whole")
            items.append((tile, kb0, kb1, kind))
    items += [(t, 0, num_kb, "whole") for t in range(sk + unit, total_tiles, units)]
    return items


def tile_rows(M: int, Ns, pairs: int, can_split: bool) -> int:
    """The activation rows per tile the launcher picks (256, 192 or 128)."""
    wtiles = sum((n + 255) // 256 for n in Ns)
    best, best_cost = 256, None
    for bn in (256, 192, 128):
        tiles = -(-M // bn) * wtiles
        split = can_split and bn == 256 and split_pays(tiles, pairs)
        waves = tiles / pairs if split else -(-tiles // pairs)
        cost = waves * (bn + 96)
        if best_cost is None or cost < best_cost:
            best, best_cost = bn, cost
    return best
