"""Index arithmetic of the decode kernel's work split, checked on the host by
enumeration.

The persistent decode grid gives warp w the units [w*W/NW, (w+1)*W/NW) of the W
units (U per (batch, KV head)); the warp writes one partial per head it touches,
at slot w - first(head), where first(head) is the first warp whose range holds the
head's first unit.  The workspace holds pmax = ceil(U / q) + 1 slots per query
head, q = floor(W / NW) (kivi_decode_splits).  A slot outside [0, pmax) would be
written outside its row, or past the workspace for the last heads: these tests
walk every warp of many splits and check that no slot leaves the row, and that
the combine's count of partials (last - first + 1) is exactly the number of warps
that touch the head.
"""
import itertools

import pytest


def owner_warp(u, W, NW):
    """First warp whose unit range holds unit u (the kernel's owner_warp)."""
    return ((u + 1) * NW - 1) // W


def pmax_of(U, W, NW):
    q = W // NW
    return (U + q - 1) // q + 1


def walk(heads, U, nw_device):
    W = heads * U
    NW = min(nw_device, W)
    pmax = pmax_of(U, W, NW)
    touched = {}
    for w in range(NW):
        u0, u1 = w * W // NW, (w + 1) * W // NW
        assert u0 < u1, "every warp of the grid holds a unit"
        for h in range(u0 // U, (u1 - 1) // U + 1):
            slot = w - owner_warp(h * U, W, NW)
            assert 0 <= slot < pmax, (heads, U, nw_device, w, h, slot, pmax)
            touched.setdefault(h, []).append(w)
    for h, ws in touched.items():
        first, last = owner_warp(h * U, W, NW), owner_warp(h * U + U - 1, W, NW)
        assert ws == list(range(first, last + 1)), (h, ws, first, last)
    assert sorted(touched) == list(range(heads))
    return pmax


@pytest.mark.parametrize("heads,U,nw", list(itertools.product([1, 2, 3, 7, 64, 256], [1, 2, 5, 65, 129, 513],
                                                              [1, 4, 456, 1824])))
def test_partial_slots_stay_in_their_rows(heads, U, nw):
    walk(heads, U, nw)


def test_workload_shapes():
    # the five workloads' splits on a 152-SM grid of 3 CTAs x 4 warps per SM, and the
    # long single-head contexts of the allocation-free entry point's test
    nw = 152 * 3 * 4
    shapes = [(1, 16), (256, 65 + 1), (128, 513 + 1), (2048, 129 + 1), (32, 4097 + 1), (1, 2001), (4, 11)]
    for heads, U in shapes:
        walk(heads, U, nw)


# ---- the small-context path: one CTA, or a cluster of CL CTAs, per (batch, KV head)

def walk_small(U, CL, NWARPS, R, kD=128):
    """The small path's split and merge addressing for one (batch, KV head) of U units
    on CL CTAs of NWARPS warps: warp `warp` of cluster CTA `rank` is gw = rank * NWARPS
    + warp and takes units [gw*U/NW, (gw+1)*U/NW), NW = min(U, CL * NWARPS).  It writes
    its partial of query head r into its own CTA's region, row warp * R + r of kD + 2
    floats (NWARPS * R rows); the first CTA's warp r reads partial j of head r from CTA
    j // NWARPS, row (j % NWARPS) * R + r.  Every unit is taken exactly once, every
    warp gw < NW takes one (at most 16 units: exactly one), no row leaves its CTA's
    region, and the merge reads exactly the rows the warps wrote."""
    NW = min(U, CL * NWARPS)
    region = NWARPS * R * (kD + 2)
    taken, written = [], set()
    for rank in range(CL):
        for warp in range(NWARPS):
            gw = rank * NWARPS + warp
            if gw >= NW:
                continue
            u0, u1 = gw * U // NW, (gw + 1) * U // NW
            assert u0 < u1, (U, CL, NWARPS, gw)
            if U <= CL * NWARPS:
                assert u1 - u0 == 1
            taken.extend(range(u0, u1))
            for r in range(R):
                off = (warp * R + r) * (kD + 2)
                assert 0 <= off and off + kD + 2 <= region
                written.add((rank, off))
    assert taken == list(range(U))
    for r in range(R):
        read = {(j // NWARPS, ((j % NWARPS) * R + r) * (kD + 2)) for j in range(NW)}
        assert read <= written and len(read) == NW
    return NW


@pytest.mark.parametrize("R", [1, 2, 4])
def test_small_and_cluster_paths(R):
    # one CTA of 8 warps up to 8 units; clusters of 4 x 4 and 2 x 8 warps for 9 to 16
    for U in range(1, 9):
        walk_small(U, 1, 8, R)
    for U in range(9, 17):
        walk_small(U, 4, 4, R)
        walk_small(U, 2, 8, R)
