"""Pins for the oracle's scale repack (CPU only).

* The layout equals the pages' logical shape [32, 4, rest_m, 4, rest_k] laid
  out atom by atom, expressed here with torch reshape/permute instead of index
  arithmetic.
* Page 1's producer address arithmetic (golden/sf_atom_addressing.json) finds
  the right 2048-byte slab for a (row tile, k-tile).
* Page 1's sfb_lane column offset (golden/sf_tmem_columns.json) selects rows
  64..127 of an atom.
* An inverse permutation recovers the input; padding is zero.
"""
import json
import os

import numpy as np
import pytest
import torch

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def rand_sf(rows, K, L=1, seed=0):
    g = torch.Generator().manual_seed(seed)
    return torch.randint(1, 256, (L, rows, K // 16), dtype=torch.uint8, generator=g)


def torch_layout(sf, rows, K):
    """[rows, K/16] -> memory order [rest_m][rest_k][r0][r1][c0] via views."""
    rm = -(-rows // 128)
    rk = -(-K // 256) * 4
    pad = torch.zeros(rm * 128, rk * 4, dtype=torch.uint8)
    pad[:rows, :K // 16] = sf
    # row = rm*128 + r1*32 + r0 ; col = ck*4 + c0
    t = pad.reshape(rm, 4, 32, rk, 4)                  # (rm, r1, r0, ck, c0)
    t = t.permute(0, 3, 2, 1, 4).contiguous()         # (rm, ck, r0, r1, c0)
    return t.reshape(-1).numpy()


@pytest.mark.parametrize("rows,K", [(128, 256), (200, 512), (1, 256), (384, 1024), (130, 768), (64, 320)])
def test_layout_matches_logical_shape(rows, K):
    sf = rand_sf(rows, K)[0]
    out = oracle.repack_scales(sf, rows, K)
    assert out.size == oracle.repacked_bytes(rows, K)
    assert np.array_equal(out, torch_layout(sf, rows, K))


def test_batches_stack_outermost():
    rows, K, L = 150, 512, 3
    sf = rand_sf(rows, K, L, seed=4)
    out = oracle.repack_scales(sf, rows, K, L)
    per = oracle.repacked_bytes(rows, K)
    for l in range(L):
        assert np.array_equal(out[l * per:(l + 1) * per], oracle.repack_scales(sf[l], rows, K))


def test_page_one_slab_addressing():
    spec = json.load(open(os.path.join(GOLDEN, "sf_atom_addressing.json")))
    for c in spec["cases"]:
        rows, K, tile, it = c["rows"], c["K"], c["tile"], c["iter_k"]
        sf = rand_sf(rows, K, seed=rows + K)[0]
        out = oracle.repack_scales(sf, rows, K)
        slab = out[c["byte_offset"]:c["byte_offset"] + c["slab_bytes"]]
        expect = sf[tile * 128:(tile + 1) * 128, it * 16:(it + 1) * 16].numpy()
        # the slab holds exactly this block of scales (as a multiset per atom)
        for a in range(4):
            atom = slab[a * 512:(a + 1) * 512]
            assert sorted(atom.tolist()) == sorted(expect[:, a * 4:(a + 1) * 4].reshape(-1).tolist())


def test_page_one_column_offset_selects_upper_rows():
    spec = json.load(open(os.path.join(GOLDEN, "sf_tmem_columns.json")))
    rows, K = 128, 256
    sf = rand_sf(rows, K, seed=9)[0].numpy()
    atom = oracle.repack_scales(sf, rows, K)[:512]
    for c in spec["cases"]:
        j = c["column_offset"]
        for r0 in range(32):
            # 32-bit column j of lane r0 = atom bytes 16*r0 + 4*j .. +3
            col = atom[16 * r0 + 4 * j:16 * r0 + 4 * j + 4]
            assert np.array_equal(col, sf[c["first_row"] + r0, 0:4])


@pytest.mark.parametrize("rows,K,L", [(300, 1024, 2), (7, 256, 1), (129, 2304, 1)])
def test_inverse_permutation_round_trip(rows, K, L):
    sf = rand_sf(rows, K, L, seed=rows)
    out = oracle.repack_scales(sf, rows, K, L)
    rm = -(-rows // 128)
    rk = -(-K // 256) * 4
    t = out.reshape(L, rm, rk, 32, 4, 4)               # (l, rm, ck, r0, r1, c0)
    back = t.transpose(0, 1, 4, 3, 2, 5).reshape(L, rm * 128, rk * 4)
    assert np.array_equal(back[:, :rows, :K // 16], sf.numpy())
    assert not back[:, rows:, :].any()
    assert not back[:, :, K // 16:].any()
