"""paged_rope_cache_write (the rotary embedding + paged KV-cache write that
runs ahead of decode) against its fp64 oracle, through the C ABI.

Bounds: a rotated value is an fp32 computation rounded once to the input
dtype, so it may differ from the exact fp64 result by half a unit in the
last place (2^-8 of the value for bf16, 2^-11 for fp16) plus the fp32
arithmetic (2^-22 of |x1| + |x2|); v is copied bit for bit; every cache
slot the call does not name keeps its bits.  Then the composition: a decode
call over the cache just written sees the new tokens (checked against the
attention oracle on the written inputs)."""

import dataclasses

import numpy as np
import pytest
import torch

import oracle
from oracle import rope_cache as R
import paged_split_kv_02_gb300 as pd
from paged_split_kv_02_gb300 import workloads as W
from gpu_helpers import check, scratch_for

pytestmark = pytest.mark.gpu

HALF_ULP = {torch.bfloat16: 2.0 ** -8, torch.float16: 2.0 ** -11}


@pytest.fixture(scope="module", autouse=True)
def _built():
    pd.build()
    pd.paged_decode_device_status(reset=True)
    yield
    assert pd.paged_decode_device_status(reset=True) == 0


def _pair_magnitude(x, rot, neox):
    """|x1| + |x2| of the pair each dim belongs to (0 past rot_dim)."""
    a, b = R.pair_index(rot, neox)
    m = np.zeros_like(x)
    s = np.abs(x[..., a]) + np.abs(x[..., b])
    m[..., a] = s
    m[..., b] = s
    return m


def _assert_rotated(gpu, ref, x_in, rot, neox, dtype, what):
    g = gpu.double().cpu().numpy()
    eps = 2.0 ** -22 * _pair_magnitude(x_in, rot, neox)
    tol = HALF_ULP[dtype] * (np.abs(ref) + eps) + eps + 2.0 ** -24
    bad = np.abs(g - ref) > tol
    assert not bad.any(), (f"{what}: {int(bad.sum())} values off, worst "
                           f"{float(np.max(np.abs(g - ref) - tol)):.3g} over the bound")


def _run_and_check(c, inplace=False):
    g = c.to("cuda")
    k0 = g.k_cache.clone()
    v0 = g.v_cache.clone()
    q_out = g.q if inplace else torch.empty_like(g.q)
    q_in = c.q.clone()
    pd.rope_case(g, q_out=q_out)
    torch.cuda.synchronize()
    assert pd.paged_decode_device_status(reset=True) == 0
    q_ref, k_pool, v_pool, written = R.rope_cache_write(
        q_in, c.k, c.v, c.positions, c.slot_mapping, c.cos_sin, c.k_cache, c.v_cache, c.layout,
        c.rot_dim, c.is_neox)
    _assert_rotated(q_out, q_ref, q_in.double().numpy(), c.rot_dim, c.is_neox, c.dtype, "q")
    # the cache: written slots rotated (k) or copied (v); the rest untouched
    nhd = c.layout == W.NHD
    kc, vc = g.k_cache.cpu(), g.v_cache.cpu()
    touched = np.zeros(kc.shape[:2] if nhd else (kc.shape[0], kc.shape[2]), dtype=bool)
    k_in = c.k.double().numpy()
    for t, page, off in written:
        touched[page, off] = True
        gk = kc[page, off] if nhd else kc[page, :, off]
        gv = vc[page, off] if nhd else vc[page, :, off]
        rk = k_pool[page, off] if nhd else k_pool[page, :, off]
        _assert_rotated(gk, rk, k_in[t], c.rot_dim, c.is_neox, c.dtype, f"k of token {t}")
        assert torch.equal(gv, c.v[t]), f"v of token {t} not copied bit for bit"
    k0c, v0c = k0.cpu(), v0.cpu()
    for page in range(touched.shape[0]):
        for off in range(touched.shape[1]):
            if touched[page, off]:
                continue
            sl = (page, off) if nhd else (page, slice(None), off)
            assert torch.equal(kc[sl], k0c[sl]) and torch.equal(vc[sl], v0c[sl]), (page, off)
    return g, q_out


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float16])
@pytest.mark.parametrize("neox", [True, False])
@pytest.mark.parametrize("D,rot", [(64, 64), (128, 128), (128, 64), (256, 64), (512, 512),
                                   (256, 256)])
def test_rope_cache_write_matches_oracle(dtype, neox, D, rot):
    c = W.make_rope_case(f"rope_{D}_{rot}", seed=D + rot, dtype=dtype, num_tokens=37,
                         num_q_heads=8, num_kv_heads=2, head_size=D, rot_dim=rot,
                         page_size=16, num_pages=5, layout=W.HND, is_neox=neox, max_pos=3000,
                         pad_tokens=3)
    _run_and_check(c)


@pytest.mark.parametrize("layout", [W.NHD, W.HND])
@pytest.mark.parametrize("packed", [False, True])
def test_rope_cache_layouts_and_packed_pool(layout, packed):
    c = W.make_rope_case("rope_layout", seed=7, dtype=torch.bfloat16, num_tokens=50,
                         num_q_heads=32, num_kv_heads=8, head_size=128, rot_dim=128,
                         page_size=16, num_pages=4, layout=layout, packed=packed, pad_tokens=5)
    _run_and_check(c)


@pytest.mark.parametrize("neox", [True, False])
@pytest.mark.parametrize("inplace", [False, True])
def test_rope_many_tokens(neox, inplace):
    """Enough tokens to fill the SMs with warps (the kernel then takes one
    item per thread per pass instead of four): 1400 tokens, partial rotary."""
    c = W.make_rope_case("rope_many", seed=13, dtype=torch.bfloat16, num_tokens=1400,
                         num_q_heads=32, num_kv_heads=8, head_size=128, rot_dim=96 if neox else 64,
                         page_size=16, num_pages=100, layout=W.HND, is_neox=neox, max_pos=4096,
                         pad_tokens=7)
    _run_and_check(c, inplace=inplace)


def test_rope_in_place_and_hybrid_page():
    # q_out = q, a 784-token page, 16 q / 2 kv heads at D = 256, 64 rotary dims
    c = W.make_rope_case("rope_inplace", seed=9, dtype=torch.bfloat16, num_tokens=64,
                         num_q_heads=16, num_kv_heads=2, head_size=256, rot_dim=64,
                         page_size=784, num_pages=2, layout=W.HND)
    _run_and_check(c, inplace=True)


def test_rope_out_of_range_position_and_slot_reported():
    c = W.make_rope_case("rope_bad", seed=11, dtype=torch.float16, num_tokens=8, num_q_heads=4,
                         num_kv_heads=2, head_size=64, rot_dim=64, page_size=16, num_pages=2,
                         max_pos=100)
    pos = c.positions.clone()
    pos[2] = 100      # past the table: clamped to its last row
    pos[3] = -4       # before it: clamped to row 0
    slots = c.slot_mapping.clone()
    slots[5] = 2 * 16  # past the pool: not written
    bad = dataclasses.replace(c, positions=pos, slot_mapping=slots)
    g = bad.to("cuda")
    k0 = g.k_cache.clone()
    q_out = pd.rope_case(g)
    torch.cuda.synchronize()
    st = pd.paged_decode_device_status(reset=True)
    assert st & pd.DEV_BAD_POSITION and st & pd.DEV_BAD_SLOT
    clamped = dataclasses.replace(bad, positions=pos.clamp(0, 99),
                                  slot_mapping=torch.where(slots >= 32, -1, slots))
    q_ref, k_pool, _, written = R.rope_cache_write(
        clamped.q, clamped.k, clamped.v, clamped.positions, clamped.slot_mapping,
        clamped.cos_sin, clamped.k_cache, clamped.v_cache, clamped.layout, clamped.rot_dim,
        clamped.is_neox)
    _assert_rotated(q_out, q_ref, c.q.double().numpy(), 64, True, torch.float16, "q")
    assert len(written) == 7
    for t, page, off in written:
        _assert_rotated(g.k_cache[page, :, off], k_pool[page, :, off], c.k.double().numpy()[t],
                        64, True, torch.float16, f"k {t}")
    # nothing else of the pool changed
    mask = torch.ones(2, 16, dtype=torch.bool)
    for _, page, off in written:
        mask[page, off] = False
    assert torch.equal(g.k_cache.permute(0, 2, 1, 3)[mask.cuda()],
                       k0.permute(0, 2, 1, 3)[mask.cuda()])


@pytest.mark.parametrize("early", [0, 1])
def test_rope_then_decode_sees_the_new_tokens(early):
    """The M new tokens of every sequence of a decode batch: rotate q and k,
    write k and v into their cache slots, then decode over that cache.  With
    early reads the decode streams the older pages while the rotary kernel
    still runs, and must wait for it before the newest keys and q."""
    M = 4
    lens = [1500, 37, 900] if not early else [6000, 37, 900, 2051]
    case = W.make_case("rope_then_decode", seed=21 + early, dtype=torch.bfloat16, head_size=128,
                       num_q_heads=32, num_kv_heads=8, page_size=16, max_query_len=M,
                       seq_lens=lens, layout=W.HND)
    S, P, Hkv, D = case.num_seqs, case.page_size, case.num_kv_heads, case.head_size
    # slots and positions of the last M tokens of every sequence
    slots, positions = [], []
    for s, L in enumerate(case.seq_lens_host):
        for k in range(L - M, L):
            phys = int(case.block_table[s, k // P])
            slots.append(phys * P + k % P)
            positions.append(k)
    T = S * M
    gen = torch.Generator().manual_seed(5)
    k_new = torch.randn(T, Hkv, D, generator=gen).to(case.dtype)
    v_new = torch.randn(T, Hkv, D, generator=gen).to(case.dtype)
    table = W.rope_cos_sin_table(8192, D)
    g = case.to("cuda")
    q_rot = torch.empty_like(g.q)
    pd.paged_rope_cache_write(g.q, k_new.cuda(), v_new.cuda(),
                              torch.tensor(positions, dtype=torch.int32, device="cuda"),
                              torch.tensor(slots, dtype=torch.int32, device="cuda"),
                              table.cuda(), q_rot, g.k_cache, g.v_cache, 32, Hkv, D, D, P,
                              W.HND, True)
    sc = scratch_for(case)
    out = pd.decode_case(dataclasses.replace(g, q=q_rot), scratch=sc,
                         opts=pd.options(early_reads=1) if early else None)
    torch.cuda.synchronize()
    assert pd.paged_decode_device_status(reset=True) == 0
    # the rope step against its oracle ...
    q_ref, k_pool, v_pool, _ = R.rope_cache_write(
        case.q, k_new, v_new, torch.tensor(positions), torch.tensor(slots), table,
        case.k_cache, case.v_cache, W.HND, D, True)
    _assert_rotated(q_rot, q_ref, case.q.double().numpy(), D, True, case.dtype, "q")
    # ... and the decode over what it wrote against the attention oracle
    written = dataclasses.replace(case, q=q_rot.cpu(), k_cache=g.k_cache.cpu(),
                                  v_cache=g.v_cache.cpu())
    check(written, out)
    # the cache the decode read holds the oracle's new tokens
    assert np.allclose(g.k_cache.double().cpu().numpy(), k_pool, rtol=2.0 ** -7, atol=1e-6,
                       equal_nan=True)
    assert np.array_equal(g.v_cache.double().cpu().numpy(), v_pool, equal_nan=True)
