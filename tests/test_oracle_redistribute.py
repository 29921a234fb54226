"""Pins for the oracle's redistribute (CPU only).

Pinned by: round-trip identities (Shard -> Replicate -> Shard,
Shard(0) -> Shard(1) -> Shard(0), Replicate -> Partial -> Replicate),
composition (A -> B -> C equals A -> C), a scalar brute-force model of the
Partial sum that finds each element's owners one by one, the fp64 bound on
the in-order fp32 sum, and the 2x2-mesh values that follow from the printed
``distribute_tensor`` example of the Hyper-Parallel DTensor API.
"""
import random

import numpy as np
import pytest

from oracle import bf16
from oracle import placement as pl
from oracle import redistribute as rd

from test_oracle_placement import random_layout


def int_valued_bf16(shape, rng):
    # small integers are exact in bf16 and their sums (|s| < 256) are exact in fp32
    v = rng.integers(-8, 9, size=shape).astype(np.float32)
    return bf16.round_rne(v)


def layouts_same_shape(rng, gshape, mesh):
    nd = len(gshape)
    pls = []
    for _ in mesh:
        r = rng.random()
        if r < 0.5:
            pls.append(pl.Shard(rng.randrange(nd)))
        elif r < 0.8:
            pls.append(pl.Replicate())
        else:
            pls.append(pl.Partial())
    return pl.Layout(mesh, pls, gshape, materialize_replicas=rng.random() < 0.25)


def test_worked_2x2_mesh_values():
    """[Shard(0), Replicate()] -> [Replicate(), Shard(1)] -> back, on arange(16).

    After the move, tp coordinate 0 holds columns 0-1 and tp coordinate 1
    columns 2-3 of the global tensor, on both dp coordinates.
    """
    g = np.arange(16, dtype=np.float32).reshape(4, 4)
    a = pl.Layout((2, 2), [pl.Shard(0), pl.Replicate()], (4, 4))
    b = pl.Layout((2, 2), [pl.Replicate(), pl.Shard(1)], (4, 4))
    la = rd.distribute(g, a, "fp32")
    lb = rd.redistribute(la, a, b, "fp32")
    assert b.nslots == 2
    for rank in range(4):
        tp = rank % 2
        np.testing.assert_array_equal(lb[b.slot_of_rank(rank)], g[:, 2 * tp:2 * tp + 2])
    back = rd.redistribute(lb, b, a, "fp32")
    for s in range(a.nslots):
        np.testing.assert_array_equal(back[s], la[s])


@pytest.mark.parametrize("seed", range(6))
def test_round_trips_and_composition(seed):
    rng = random.Random(seed)
    nrng = np.random.default_rng(seed)
    for _ in range(40):
        nm = rng.randint(1, 3)
        mesh = tuple(rng.randint(1, 3) for _ in range(nm))
        gshape = tuple(rng.randint(1, 7) for _ in range(rng.randint(1, 3)))
        g = int_valued_bf16(gshape, nrng)
        a = layouts_same_shape(rng, gshape, mesh)
        b = layouts_same_shape(rng, gshape, mesh)
        c = layouts_same_shape(rng, gshape, mesh)
        # start from a Replicate-derived source so every layout is legal
        rep = pl.Layout(mesh, [pl.Replicate()] * nm, gshape)
        la = rd.redistribute([g], rep, a, "bf16")
        np.testing.assert_array_equal(rd.to_global(la, a, "bf16"), g)

        def move(lx, x, y):
            try:
                return rd.redistribute(lx, x, y, "bf16")
            except NotImplementedError:
                return None

        lb = move(la, a, b)
        if lb is None:
            continue
        np.testing.assert_array_equal(rd.to_global(lb, b, "bf16"), g)
        lc_via_b = move(lb, b, c)
        lc_direct = move(la, a, c)
        if lc_via_b is None or lc_direct is None:
            continue
        np.testing.assert_array_equal(rd.to_global(lc_via_b, c, "bf16"), g)
        # composition: a -> b -> c and a -> c agree slot by slot where b keeps
        # no Partial that c also keeps (then partial splits may differ)
        if not any(isinstance(b.placements[m], pl.Partial) and isinstance(c.placements[m], pl.Partial)
                   for m in range(nm)):
            for s in range(c.nslots):
                np.testing.assert_array_equal(lc_via_b[s], lc_direct[s])
        # back to a: identity when a holds no Partial
        if not a.partial_dims():
            back = move(lc_direct, c, a)
            if back is not None:
                for s in range(a.nslots):
                    np.testing.assert_array_equal(back[s], la[s])


def brute_force_reduce(locals_, layout, index):
    """Scalar model: visit every rank, keep those whose block holds ``index``,
    add their values in rank order in fp32 (first value taken as is)."""
    acc = None
    seen_slots = set()
    for rank in range(pl.mesh_size(layout.mesh_shape)):
        coords = pl.rank_coords(layout.mesh_shape, rank)
        if any(coords[m] != 0 for m, p in enumerate(layout.placements) if isinstance(p, pl.Replicate)):
            continue
        box = layout.box_of_coords(coords)
        if not all(o <= i < o + s for (o, s), i in zip(box, index)):
            continue
        slot = layout.slot_of_coords(coords)
        assert slot not in seen_slots
        seen_slots.add(slot)
        local_idx = tuple(i - o for (o, _), i in zip(box, index))
        v = np.float32(bf16.widen(np.array([locals_[slot][local_idx]], dtype=np.uint16))[0])
        acc = v if acc is None else np.float32(acc + v)
    return acc


def check_partial_sum_brute_force(redistribute=rd):
    nrng = np.random.default_rng(5)
    mesh = (2, 3)
    gshape = (5, 7)
    src = pl.Layout(mesh, [pl.Partial(), pl.Shard(1)], gshape)
    dst = pl.Layout(mesh, [pl.Replicate(), pl.Replicate()], gshape)
    locals_ = [bf16.round_rne(nrng.standard_normal(src.local_shape(s)).astype(np.float32) * 10.0 ** nrng.integers(-3, 4))
               for s in range(src.nslots)]
    out = redistribute.redistribute(locals_, src, dst, "bf16")[0]
    for i in range(gshape[0]):
        for j in range(gshape[1]):
            acc = brute_force_reduce(locals_, src, (i, j))
            assert out[i, j] == bf16.round_rne(np.array([acc], dtype=np.float32))[0], (i, j)


def test_partial_sum_matches_scalar_brute_force():
    check_partial_sum_brute_force()


def test_partial_sum_order_is_rank_order():
    # fp32: ((1e8 + 1) - 1e8) + 1 = 1 in rank order; other orders give 0 or 2.
    mesh = (4,)
    src = pl.Layout(mesh, [pl.Partial()], (1,))
    dst = pl.Layout(mesh, [pl.Replicate()], (1,))
    vals = [np.array([v], dtype=np.float32) for v in (1e8, 1.0, -1e8, 1.0)]
    assert rd.redistribute(vals, src, dst, "fp32")[0][0] == np.float32(1.0)


def test_partial_sum_within_fp64_bound():
    nrng = np.random.default_rng(9)
    mesh = (2, 4)
    gshape = (64, 96)
    src = pl.Layout(mesh, [pl.Shard(0), pl.Partial()], gshape)
    dst = pl.Layout(mesh, [pl.Shard(0), pl.Replicate()], gshape)
    locals_ = [bf16.round_rne(nrng.standard_normal(src.local_shape(s))) for s in range(src.nslots)]
    out = rd.redistribute(locals_, src, dst, "bf16")
    for dp in range(2):
        exact = sum(bf16.widen64(locals_[src.slot_of_coords((dp, t))]) for t in range(4))
        got = bf16.widen64(out[dst.slot_of_coords((dp, 0))])
        # half an ulp of bf16 plus three fp32 roundings of partial sums
        mag = sum(np.abs(bf16.widen64(locals_[src.slot_of_coords((dp, t))])) for t in range(4))
        bound = np.abs(exact) * 2.0 ** -8 + 3 * mag * 2.0 ** -24 + 1e-30
        assert (np.abs(got - exact) <= bound).all()


def test_replicate_to_partial_keeps_value_at_zero():
    g = np.arange(12, dtype=np.float32).reshape(3, 4)
    rep = pl.Layout((3,), [pl.Replicate()], (3, 4))
    par = pl.Layout((3,), [pl.Partial()], (3, 4))
    lp = rd.redistribute([g], rep, par, "fp32")
    np.testing.assert_array_equal(lp[0], g)
    assert not lp[1].any() and not lp[2].any()
    np.testing.assert_array_equal(rd.redistribute(lp, par, rep, "fp32")[0], g)


def test_shard_to_partial_is_rejected():
    a = pl.Layout((2,), [pl.Shard(0)], (4, 4))
    b = pl.Layout((2,), [pl.Partial()], (4, 4))
    with pytest.raises(NotImplementedError):
        rd.redistribute([np.zeros((2, 4), np.float32)] * 2, a, b, "fp32")


def test_partial_to_shard0_is_reduce_scatter():
    nrng = np.random.default_rng(3)
    mesh = (4,)
    src = pl.Layout(mesh, [pl.Partial()], (10, 6))
    dst = pl.Layout(mesh, [pl.Shard(0)], (10, 6))
    locals_ = [bf16.round_rne(nrng.standard_normal((10, 6))) for _ in range(4)]
    full = rd.redistribute(locals_, src, pl.Layout(mesh, [pl.Replicate()], (10, 6)), "bf16")[0]
    parts = rd.redistribute(locals_, src, dst, "bf16")
    np.testing.assert_array_equal(np.concatenate(parts, axis=0), full)
    assert [p.shape[0] for p in parts] == [3, 3, 3, 1]


def test_planted_sum_order_mistake_is_caught(monkeypatch):
    """Adding partials in reverse rank order must fail the brute-force pin."""
    orig = rd.to_global

    def reversed_order(locals_, layout, dtype, keep=None):
        if layout.partial_dims():
            # reverse the stored partial slots along the partial dim
            perm = []
            for s in range(layout.nslots):
                c = list(layout.slot_coords(s))
                for m in layout.partial_dims():
                    c[m] = layout.mesh_shape[m] - 1 - c[m]
                perm.append(layout.slot_of_coords(c))
            locals_ = [locals_[perm[s]] for s in range(layout.nslots)]
        return orig(locals_, layout, dtype, keep)

    monkeypatch.setattr(rd, "to_global", reversed_order)
    with pytest.raises(AssertionError):
        test_partial_sum_order_is_rank_order()


def test_partial_avg_and_max_brute_force():
    """Partial(avg): rank-order fp32 sum, one fp32 division, one bf16 rounding;
    Partial(max): rank-order maximum -- checked against scalar loops."""
    nrng = np.random.default_rng(21)
    mesh = (2, 3)
    gshape = (4, 7)
    for op in ("avg", "max"):
        src = pl.Layout(mesh, [pl.Partial(op), pl.Shard(1)], gshape)
        dst = pl.Layout(mesh, [pl.Replicate(), pl.Replicate()], gshape)
        locals_ = [bf16.round_rne(nrng.standard_normal(src.local_shape(s)) * 7.0) for s in range(src.nslots)]
        out = rd.redistribute(locals_, src, dst, "bf16")[0]
        for i in range(gshape[0]):
            for j in range(gshape[1]):
                vals = []
                for c0 in range(2):  # rank order over the Partial dim
                    c = (c0, None)
                    for c1 in range(3):
                        box = src.box_of_coords((c0, c1))
                        (o0, s0), (o1, s1) = box
                        if o1 <= j < o1 + s1:
                            v = bf16.widen(np.array([locals_[src.slot_of_coords((c0, c1))][i - o0, j - o1]]))[0]
                            vals.append(np.float32(v))
                if op == "avg":
                    acc = vals[0]
                    for v in vals[1:]:
                        acc = np.float32(acc + v)
                    ref = np.float32(acc / np.float32(len(vals)))
                else:
                    ref = vals[0]
                    for v in vals[1:]:
                        ref = v if v > ref else ref
                assert out[i, j] == bf16.round_rne(np.array([ref], dtype=np.float32))[0], (op, i, j)


def test_partial_avg_max_round_trips_and_closed_forms():
    g = np.arange(24, dtype=np.float32).reshape(4, 6)
    for op in ("avg", "max"):
        rep = pl.Layout((4,), [pl.Replicate()], (4, 6))
        par = pl.Layout((4,), [pl.Partial(op)], (4, 6))
        lp = rd.redistribute([g], rep, par, "fp32")
        assert all(np.array_equal(x, g) for x in lp)          # every coordinate keeps the value
        np.testing.assert_array_equal(rd.redistribute(lp, par, rep, "fp32")[0], g)
    # avg of 4 partials 1, 2, 3, 6 is 3; max is 6; sum is 12
    vals = [np.full((1,), v, np.float32) for v in (1.0, 2.0, 3.0, 6.0)]
    for op, want in (("sum", 12.0), ("avg", 3.0), ("max", 6.0)):
        src = pl.Layout((4,), [pl.Partial(op)], (1,))
        assert rd.redistribute(vals, src, pl.Layout((4,), [pl.Replicate()], (1,)), "fp32")[0][0] == want
    with pytest.raises(NotImplementedError):
        rd.redistribute(vals, pl.Layout((4,), [pl.Partial("avg")], (1,)), pl.Layout((4,), [pl.Partial("max")], (1,)),
                        "fp32")
