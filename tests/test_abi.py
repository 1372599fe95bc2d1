"""Host-side checks of the C ABI: the library loads without a GPU, exports every
declared symbol, plans deterministically, and rejects bad arguments before any
CUDA call (every case here fails validation, so nothing is launched)."""
import ctypes
import math
import os
import re

import pytest

import decode_attention_mla_gb300 as mla
from decode_attention_mla_gb300 import build as mla_build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SCALE = 1.0 / math.sqrt(576)


@pytest.fixture(scope="module", autouse=True)
def built():
    mla_build.build()
    yield


def _declared_symbols():
    names = set()
    for fn in os.listdir(os.path.join(ROOT, "include")):
        if fn.endswith(".h"):
            text = open(os.path.join(ROOT, "include", fn)).read()
            names |= set(re.findall(r"MLA_API\s+[\w\s\*]+?\b(mla_\w+)\s*\(", text))
    return names


def test_library_exports_every_declared_symbol():
    names = _declared_symbols()
    assert names, "no declarations found"
    assert set(mla.EXPORTED) <= names
    L = ctypes.CDLL(mla.LIB_PATH)
    for n in sorted(names):
        assert hasattr(L, n), f"{n} declared but not exported"
    assert mla.abi_version() == 4
    assert "scratch" in mla.strerror(mla.ESCRATCH)


def _plan(**kw):
    base = dict(batch=1, heads=16, scale=SCALE, num_sms=152)
    base.update(kw)
    return mla.plan(**base)


TILE = {1: 32, 2: 80, 3: 64, 4: 64}     # rows per modelled step: warp-MMA slot, tcgen05 tiles (16 / 32 / 64 heads)
GRANULE = {1: 32, 2: 16, 3: 16, 4: 16}  # slices are whole multiples of this
HEADS = {1: 16, 2: 16, 3: 32, 4: 64}    # heads per CTA


def _model_split(rows, pairs, sms, variant=2, max_splits=256):
    """The planner's split rule, evaluated independently: minimise
    ceil(items / grid) * (tiles per slice + 1), smallest S on ties."""
    tile, gran = TILE[variant], GRANULE[variant]
    best = None
    for S in range(1, min(max_splits, -(-rows // gran)) + 1):
        per = -(-(-(-rows // S)) // gran) * gran
        items = pairs * -(-rows // per)
        waves = -(-items // min(items, sms))
        cost = waves * (-(-per // tile) + 1)
        if best is None or cost < best[0]:
            best = (cost, S)
    return best[1]


@pytest.mark.parametrize("kw,variant,splits,entries", [
    (dict(max_ctx=256), 1, 8, 32),
    (dict(max_ctx=8192), 1, 128, 64),
    (dict(sparse=True, topk=2048), 1, 64, 32),
    (dict(batch=64, sparse=True, topk=2048), 1, 4, 864),         # flat split: 152 ranges of 864 entries
    (dict(heads=128, max_ctx=32768 + 64), 4, 74, 448),
    (dict(heads=128, max_ctx=32768 + 64, variant=3), 3, 37, 896),
    (dict(heads=64, max_ctx=32768), 4, 128, 256),
    (dict(max_ctx=131072), 1, 152, 864),
    (dict(max_ctx=131072, variant=2), 2, 149, 880),
    (dict(heads=32, max_ctx=32768), 1, 74, 448),
    (dict(heads=32, max_ctx=131072), 3, 147, 896),
    (dict(max_ctx=8192, variant=2), 2, 103, 80),
    (dict(sparse=True, topk=2048, variant=2), 2, 26, 80),
    (dict(batch=64, sparse=True, topk=2048, variant=2), 2, 2, 1024),
])
def test_plan_derivation_for_the_workloads(kw, variant, splits, entries):
    p = _plan(**kw)
    assert (p.variant, p.splits, p.entries_per_split) == (variant, splits, entries)
    rows = kw.get("topk") or kw.get("max_ctx")
    B, H = kw.get("batch", 1), kw.get("heads", 16)
    if not p.flat_ranges:
        assert p.splits * p.entries_per_split >= rows
        assert (p.splits - 1) * p.entries_per_split < rows + p.entries_per_split
    assert p.n_head_groups == H // HEADS[variant] and p.ctas_per_sm == 1
    if p.flat_ranges:
        assert p.grid_x == p.flat_ranges * p.n_head_groups <= 152 and p.grid_y == 1 and p.grid_z == 1
    else:
        assert p.grid_x == min(B * p.n_head_groups * p.splits, 152) and p.grid_y == 1 and p.grid_z == 1
    assert p.combine_grid_x == -(-B * H // (8 // _unit_warps(p.splits))) and p.combine_grid_y == 4
    assert p.combine_block == 256
    # scratch layout: status word, then o_part, then lse_part, 256-byte aligned
    bh = B * H
    assert p.status_offset == 0 and p.o_part_offset % 256 == 0 and p.lse_part_offset % 256 == 0
    assert p.lse_part_offset >= p.o_part_offset + bh * p.splits * 512 * 4
    assert p.scratch_bytes >= p.lse_part_offset + bh * p.splits * 4 and p.scratch_bytes % 256 == 0


@pytest.mark.parametrize("rows", [1, 100, 8192, 32768, 131072])
@pytest.mark.parametrize("batch,heads", [(1, 64), (2, 64), (1, 128), (3, 128)])
def test_plan_head_group_64(rows, batch, heads):
    p = _plan(max_ctx=rows, batch=batch, heads=heads, variant=4)
    assert p.variant == 4 and p.head_group == 64 and p.n_head_groups == heads // 64
    assert p.splits == _model_split(rows, batch * heads // 64, 152, 4)
    assert p.entries_per_split == -(-(-(-rows // p.splits)) // 16) * 16
    assert p.grid_x == min(batch * (heads // 64) * p.splits, 152)
    assert p.block == 256 and p.smem_bytes <= 227 * 1024
    bad = mla.Plan.from_buffer_copy(p)
    bad.head_group = 32
    assert _call("mla_decode_run", bad, _args(row_offset=0x60000)) == mla.EINVAL


@pytest.mark.parametrize("rows", [1, 100, 8192, 131072])
@pytest.mark.parametrize("batch,heads", [(1, 32), (2, 64), (1, 128)])
def test_plan_head_group_32(rows, batch, heads):
    p = _plan(max_ctx=rows, batch=batch, heads=heads, variant=3)
    assert p.variant == 3 and p.head_group == 32 and p.n_head_groups == heads // 32
    assert p.splits == _model_split(rows, batch * heads // 32, 152, 3)
    assert p.entries_per_split == -(-(-(-rows // p.splits)) // 16) * 16
    assert p.grid_x == min(batch * (heads // 32) * p.splits, 152)
    assert p.block == 384 and p.smem_bytes <= 227 * 1024
    bad = mla.Plan.from_buffer_copy(p)
    bad.head_group = 16
    assert _call("mla_decode_run", bad, _args(row_offset=0x60000)) == mla.EINVAL


@pytest.mark.parametrize("variant", [1, 2])
@pytest.mark.parametrize("rows", [1, 31, 32, 33, 100, 256, 1000, 8192, 20000, 131072])
@pytest.mark.parametrize("batch,heads,sms", [(1, 16, 152), (1, 16, 132), (4, 16, 152), (64, 16, 152),
                                             (1, 128, 152), (3, 64, 148)])
def test_plan_split_rule_matches_model(variant, rows, batch, heads, sms):
    p = _plan(max_ctx=rows, batch=batch, heads=heads, num_sms=sms, variant=variant)
    assert p.splits == _model_split(rows, batch * heads // 16, sms, variant)
    ps = _plan(sparse=True, topk=rows, batch=batch, heads=heads, num_sms=sms, variant=variant)
    if ps.flat_ranges:   # batched sparse on the warp-MMA kernel may take the flat split instead
        assert variant == 1 and batch > 1
        assert (ps.flat_ranges, ps.entries_per_split, ps.splits) == _model_flat(rows, batch, heads // 16, sms)[:3]
    else:
        assert ps.splits == p.splits


def _model_auto(sparse, rows, batch, heads, sms):
    """The automatic kernel choice, restated: sparse or 16 heads -> warp-MMA;
    more heads -> warp-MMA while its slices hold <= 768 rows, else tcgen05
    with 64 heads per CTA (H a multiple of 64) or 32."""
    def per(v):
        S = _model_split(rows, batch * heads // HEADS[v], sms, v)
        return -(-(-(-rows // S)) // GRANULE[v]) * GRANULE[v]
    if sparse or heads == 16:
        return 1
    if per(1) <= 768:
        return 1
    return 4 if heads % 64 == 0 else 3


@pytest.mark.parametrize("rows", [1, 100, 256, 8192, 20000, 32768, 65536, 131072])
@pytest.mark.parametrize("batch,heads", [(1, 16), (4, 16), (1, 32), (1, 64), (2, 128)])
@pytest.mark.parametrize("sparse", [False, True])
def test_plan_automatic_kernel_choice(rows, batch, heads, sparse):
    kw = dict(sparse=True, topk=rows) if sparse else dict(max_ctx=rows)
    p = _plan(batch=batch, heads=heads, **kw)
    v = _model_auto(sparse, rows, batch, heads, 152)
    assert p.variant == v
    S = _model_split(rows, batch * heads // HEADS[v], 152, v)
    flat = _model_flat(rows, batch, heads // HEADS[v], 152) if (sparse and v == 1) else None
    if flat and flat[3] < _model_uniform_cost(rows, batch * heads // HEADS[v], 152, v, S):
        assert (p.flat_ranges, p.entries_per_split, p.splits) == flat[:3]
    else:
        assert p.flat_ranges == 0 and p.splits == S


def _model_uniform_cost(rows, pairs, sms, variant, S):
    tile, gran = TILE[variant], GRANULE[variant]
    per = -(-(-(-rows // S)) // gran) * gran
    items = pairs * -(-rows // per)
    return -(-items // min(items, sms)) * (-(-per // tile) + 1)


def _model_flat(topk, batch, groups, sms):
    """The flat split restated: (ranges, entries per range, most pieces per
    request, modelled cost), or None where it does not apply."""
    G = sms // groups
    if batch < 2 or G < 2:
        return None
    total = batch * topk
    per = -(-(-(-total // G)) // 32) * 32
    if per > topk:
        return None
    ranges = -(-total // per)
    s_max = max(((b + 1) * topk - 1) // per - (b * topk) // per + 1 for b in range(batch))
    return ranges, per, s_max, per // 32 + 2


def _flat_pieces(topk, batch, ranges, per):
    """The kernel's flat item coordinates, restated: for every (part, range)
    the request, slice, entries and whether the piece exists / is the last."""
    out = []
    total = batch * topk
    for part in (0, 1):
        for r in range(ranges):
            start, end = r * per, min(r * per + per, total)
            b = start // topk + part
            lo, hi = b * topk, b * topk + topk
            if start >= total or b >= batch or end <= lo:
                out.append(None)
                continue
            out.append((b, r - lo // per, max(start, lo) - lo, min(end, hi) - lo, end >= hi))
    return out


@pytest.mark.parametrize("batch,topk,sms,heads", [(64, 2048, 152, 16), (3, 700, 4, 16), (17, 96, 152, 16),
                                                  (64, 2048, 132, 32), (5, 4096, 8, 16), (2, 64, 3, 16)])
def test_plan_flat_split_covers_every_entry_once(batch, topk, sms, heads):
    """Where the planner takes the flat split, its pieces cover every list
    entry of every request exactly once, each request's pieces are its
    slices 0 .. n-1 in order, and n <= splits (the rest are written empty)."""
    p = _plan(batch=batch, heads=heads, sparse=True, topk=topk, num_sms=sms)
    model = _model_flat(topk, batch, heads // 16, sms)
    if not p.flat_ranges:
        assert model is None or model[3] >= _model_uniform_cost(
            topk, batch * heads // 16, sms, 1, _model_split(topk, batch * heads // 16, sms, 1))
        return
    assert (p.flat_ranges, p.entries_per_split, p.splits) == model[:3]
    assert p.entries_per_split % 32 == 0 and p.entries_per_split <= topk
    seen = {b: [] for b in range(batch)}
    for piece in _flat_pieces(topk, batch, p.flat_ranges, p.entries_per_split):
        if piece:
            b, s, e0, e1, last = piece
            assert 0 <= s < p.splits and e0 < e1
            seen[b].append((s, e0, e1, last))
    for b, pieces in seen.items():
        pieces.sort()
        assert [s for s, _, _, _ in pieces] == list(range(len(pieces)))
        assert pieces[0][1] == 0 and pieces[-1][2] == topk and pieces[-1][3]
        assert all(pieces[i][2] == pieces[i + 1][1] for i in range(len(pieces) - 1))
        assert sum(1 for q in pieces if q[3]) == 1


def _unit_warps(splits):
    """Warps that merge one (request, head): one lse per thread, at most 20
    slices per warp up to 8 warps, rounded up to a power of two."""
    need = max(-(-splits // 32), min(-(-splits // 20), 8))
    w = 1
    while w < need:
        w *= 2
    return w


@pytest.mark.parametrize("splits", [1, 2, 16, 17, 20, 21, 32, 33, 40, 41, 74, 80, 81, 100, 128, 149, 160, 161, 256])
@pytest.mark.parametrize("batch", [1, 3, 64])
def test_combine_grid_follows_the_split_count(splits, batch):
    p = _plan(max_ctx=131072, splits=splits, batch=batch)
    w = _unit_warps(splits)
    assert 32 * w >= splits and -(-splits // w) <= 32
    assert p.combine_block == 256
    assert p.combine_grid_x == -(-batch * 16 // (8 // w))
    bad = mla.Plan.from_buffer_copy(p)
    bad.combine_grid_x += 1
    assert _call("mla_decode_combine", bad, _args(row_offset=0x60000)) == mla.EINVAL
    bad = mla.Plan.from_buffer_copy(p)
    bad.combine_block = 128
    assert _call("mla_decode_combine", bad, _args(row_offset=0x60000)) == mla.EINVAL


def test_plan_scales_with_sm_count_and_is_deterministic():
    a = _plan(max_ctx=131072, num_sms=132, variant=2)
    b = _plan(max_ctx=131072, num_sms=132, variant=2)
    assert a.as_dict() == b.as_dict()
    assert a.splits == _model_split(131072, 1, 132) and a.grid_x <= 132
    assert _plan(max_ctx=131072, num_sms=152, variant=2).splits == _model_split(131072, 1, 152)
    assert _plan(max_ctx=131072, batch=4, num_sms=132, variant=2).splits == _model_split(131072, 4, 132)
    # short contexts: one tile per slice
    assert _plan(max_ctx=100, num_sms=152, variant=2).entries_per_split <= 80


def test_plan_override():
    for s in (1, 2, 7, 64, 128, 256):
        for v in (1, 2):
            p = _plan(max_ctx=8192, splits=s, variant=v)
            assert p.splits == s and p.grid_x == min(s, 152)
            assert p.entries_per_split == -(-(-(-8192 // s)) // GRANULE[v]) * GRANULE[v]


@pytest.mark.parametrize("kw,status", [
    (dict(heads=8, max_ctx=16), mla.EUNSUPPORTED),
    (dict(heads=48, max_ctx=16), mla.EUNSUPPORTED),
    (dict(batch=0, max_ctx=16), mla.EINVAL),
    (dict(max_ctx=0), mla.EINVAL),
    (dict(sparse=True, topk=0), mla.EINVAL),
    (dict(max_ctx=16, scale=0.0), mla.EINVAL),
    (dict(max_ctx=16, scale=float("nan")), mla.EINVAL),
    (dict(max_ctx=16, scale=float("inf")), mla.EINVAL),
    (dict(max_ctx=16, splits=257), mla.EINVAL),
    (dict(max_ctx=16, splits=-1), mla.EINVAL),
    (dict(max_ctx=16, num_sms=-5), mla.EINVAL),
    (dict(max_ctx=16, variant=7), mla.EINVAL),
    (dict(max_ctx=16, variant=6), mla.EINVAL),
    (dict(sparse=True, topk=64, variant=5), mla.EUNSUPPORTED),        # P . V on tcgen05: dense only
    (dict(max_ctx=16, heads=32, variant=4), mla.EUNSUPPORTED),         # 64 heads per CTA: H = 32 is too few
    (dict(heads=64, sparse=True, topk=64, variant=4), mla.EUNSUPPORTED),  # dense only
    (dict(max_ctx=16, variant=3), mla.EUNSUPPORTED),                 # 32 heads per CTA: H = 16 is too few
    (dict(heads=32, sparse=True, topk=64, variant=3), mla.EUNSUPPORTED),  # dense only
])
def test_plan_rejects(kw, status):
    with pytest.raises(mla.MLADecodeError) as e:
        _plan(**kw)
    assert e.value.status == status


def test_plan_rejects_bad_stall_hook():
    s = mla.Shape(batch=1, heads=16, d_latent=512, d_rope=64, sparse=0, max_ctx=16, topk=0, scale=SCALE,
                  num_sms=152, splits_override=0, variant=0, pdl=0, stall_test=2)
    assert mla.lib().mla_decode_plan(ctypes.byref(s), ctypes.byref(mla.Plan())) == mla.EINVAL
    assert _plan(max_ctx=16, stall_test=True).shape.stall_test == 1


def test_plan_rejects_bad_dims():
    L = mla.lib()
    s = mla.Shape(batch=1, heads=16, d_latent=256, d_rope=64, sparse=0, max_ctx=16, topk=0, scale=SCALE,
                  num_sms=152, splits_override=0, variant=0, pdl=0)
    p = mla.Plan()
    assert L.mla_decode_plan(ctypes.byref(s), ctypes.byref(p)) == mla.EUNSUPPORTED
    s.d_latent, s.d_rope = 512, 32
    assert L.mla_decode_plan(ctypes.byref(s), ctypes.byref(p)) == mla.EUNSUPPORTED
    assert L.mla_decode_plan(None, ctypes.byref(p)) == mla.EINVAL
    assert L.mla_decode_plan(ctypes.byref(s), None) == mla.EINVAL


def _args(**kw):
    base = dict(q=0x10000, kv=0x20000, kv_rows=100, row_stride=576, d_pos=0x30000, row_offset=None,
                cache_len=None, indices=None, out=0x40000, lse=0x50000)
    base.update(kw)
    return mla.Args(**base)


def _call(fn, p, a, scratch=0x100000, nbytes=None):
    L = mla.lib()
    nbytes = (p.scratch_bytes if p is not None else 1 << 20) if nbytes is None else nbytes
    return getattr(L, fn)(ctypes.byref(p) if p is not None else None, ctypes.byref(a) if a is not None else None,
                          ctypes.c_void_p(scratch) if scratch else None, nbytes, None)


@pytest.mark.parametrize("fn", ["mla_decode_run", "mla_decode_combine", "mla_decode_forward"])
def test_launch_argument_checks(fn):
    p = _plan(max_ctx=64)
    assert _call(fn, None, _args()) == mla.EINVAL
    bad = mla.Plan.from_buffer_copy(p)
    bad.magic = 0
    assert _call(fn, bad, _args()) == mla.EINVAL
    bad = mla.Plan.from_buffer_copy(p)
    bad.splits = 0
    assert _call(fn, bad, _args()) == mla.EINVAL
    assert _call(fn, p, None) == mla.EINVAL
    assert _call(fn, p, _args(q=None)) == mla.EINVAL
    assert _call(fn, p, _args(kv=None)) == mla.EINVAL
    assert _call(fn, p, _args(out=None)) == mla.EINVAL
    assert _call(fn, p, _args(lse=None)) == mla.EINVAL
    assert _call(fn, p, _args(d_pos=None)) == mla.EINVAL
    assert _call(fn, p, _args(kv_rows=0)) == mla.EINVAL
    assert _call(fn, p, _args(row_stride=512)) == mla.EINVAL
    assert _call(fn, p, _args(row_stride=580)) == mla.EALIGN
    assert _call(fn, p, _args(q=0x10002)) == mla.EALIGN
    assert _call(fn, p, _args(kv=0x20008)) == mla.EALIGN
    assert _call(fn, p, _args(out=0x40004)) == mla.EALIGN
    assert _call(fn, p, _args(lse=0x50002)) == mla.EALIGN
    assert _call(fn, p, _args(d_pos=0x30002)) == mla.EALIGN
    assert _call(fn, p, _args(row_offset=0x60004)) == mla.EALIGN
    # scratch checks come after the argument checks and still before any launch
    assert _call(fn, p, _args(), scratch=0) == mla.ESCRATCH
    assert _call(fn, p, _args(), scratch=0x100080) == mla.ESCRATCH
    assert _call(fn, p, _args(), nbytes=p.scratch_bytes - 1) == mla.ESCRATCH
    # dense batches > 1 need row offsets; sparse needs indices, lengths and offsets
    p2 = _plan(max_ctx=64, batch=2)
    assert _call(fn, p2, _args()) == mla.EINVAL
    ps = _plan(sparse=True, topk=64)
    assert _call(fn, ps, _args()) == mla.EINVAL
    assert _call(fn, ps, _args(indices=0x70000, cache_len=0x71000)) == mla.EINVAL
    assert _call(fn, ps, _args(indices=0x70002, cache_len=0x71000, row_offset=0x72000)) == mla.EALIGN


@pytest.mark.parametrize("fn", ["mla_decode_run", "mla_decode_combine", "mla_decode_forward"])
def test_launch_rejects_a_plan_whose_scratch_layout_is_stale(fn):
    """A plan edited to hold more slices (its grids updated to match) but whose
    scratch layout was left as planned would make the kernels write partial
    rows past the region it claims: every launch re-derives the layout."""
    p = _plan(max_ctx=8192, splits=64)
    q = _plan(max_ctx=8192, splits=128)
    bad = mla.Plan.from_buffer_copy(p)
    bad.splits, bad.grid_x, bad.combine_grid_x = q.splits, q.grid_x, q.combine_grid_x
    assert bad.scratch_bytes < q.scratch_bytes
    assert _call(fn, bad, _args(), nbytes=q.scratch_bytes) == mla.EINVAL
    for field in ("scratch_bytes", "o_part_offset", "lse_part_offset", "status_offset"):
        bad = mla.Plan.from_buffer_copy(p)
        setattr(bad, field, getattr(bad, field) + 256)
        assert _call(fn, bad, _args(), nbytes=1 << 30) == mla.EINVAL, field
    # the same edit with the layout re-derived as the planner does is a valid plan
    ok = mla.Plan.from_buffer_copy(q)
    assert _call(fn, ok, _args(), scratch=0, nbytes=q.scratch_bytes) == mla.ESCRATCH


def test_append_advance_argument_checks():
    L = mla.lib()
    assert L.mla_decode_append(None, 10, 576, ctypes.c_void_p(0x1000), ctypes.c_void_p(0x2000), None, 1, None) == mla.EINVAL
    assert L.mla_decode_append(ctypes.c_void_p(0x1000), 0, 576, ctypes.c_void_p(0x1000), ctypes.c_void_p(0x2000),
                               None, 1, None) == mla.EINVAL
    assert L.mla_decode_append(ctypes.c_void_p(0x1000), 10, 576, ctypes.c_void_p(0x1000), ctypes.c_void_p(0x2000),
                               None, 2, None) == mla.EINVAL
    assert L.mla_decode_append(ctypes.c_void_p(0x1008), 10, 576, ctypes.c_void_p(0x1000), ctypes.c_void_p(0x2000),
                               None, 1, None) == mla.EALIGN
    assert L.mla_decode_append(ctypes.c_void_p(0x1000), 10, 578, ctypes.c_void_p(0x1000), ctypes.c_void_p(0x2000),
                               None, 1, None) == mla.EALIGN
    assert L.mla_decode_advance(None, 1, None) == mla.EINVAL
    assert L.mla_decode_advance(ctypes.c_void_p(0x1000), 0, None) == mla.EINVAL
    assert L.mla_decode_advance(ctypes.c_void_p(0x1002), 1, None) == mla.EALIGN
    assert L.mla_decode_scratch_init(None, 16, None) == mla.EINVAL


def test_project_argument_checks():
    """mla_decode_project validates everything before any launch."""
    L = mla.lib()
    A, W, Y = ctypes.c_void_p(0x1000), ctypes.c_void_p(0x2000), ctypes.c_void_p(0x3000)
    assert L.mla_decode_project(None, W, 1, 16, 128, Y, 0, None) == mla.EINVAL
    assert L.mla_decode_project(A, None, 1, 16, 128, Y, 0, None) == mla.EINVAL
    assert L.mla_decode_project(A, W, 1, 16, 128, None, 0, None) == mla.EINVAL
    assert L.mla_decode_project(A, W, 0, 16, 128, Y, 0, None) == mla.EINVAL
    assert L.mla_decode_project(A, W, 1, 16, 128, Y, 2, None) == mla.EINVAL
    assert L.mla_decode_project(A, W, 1, 0, 128, Y, 0, None) == mla.EUNSUPPORTED
    assert L.mla_decode_project(A, W, 1, 129, 128, Y, 0, None) == mla.EUNSUPPORTED
    assert L.mla_decode_project(A, W, 1, 16, 120, Y, 0, None) == mla.EUNSUPPORTED
    assert L.mla_decode_project(A, W, 1, 16, 528, Y, 0, None) == mla.EUNSUPPORTED
    assert L.mla_decode_project(ctypes.c_void_p(0x1004), W, 1, 16, 128, Y, 0, None) == mla.EALIGN
    assert L.mla_decode_project(A, ctypes.c_void_p(0x2008), 1, 16, 128, Y, 0, None) == mla.EALIGN
    assert L.mla_decode_project(A, W, 1, 16, 128, ctypes.c_void_p(0x3004), 0, None) == mla.EALIGN


def test_forward_step_argument_checks():
    """mla_decode_forward_step rejects what it cannot run before any launch:
    sparse plans, a missing or misaligned new-row buffer, advance not 0/1, and
    everything mla_decode_forward rejects."""
    L = mla.lib()
    p = _plan(max_ctx=64)
    a = _args(row_offset=None)
    rows = ctypes.c_void_p(0x70000)

    def call(plan, args, new_rows, adv, scratch=0x100000, nbytes=None):
        nb = plan.scratch_bytes if (plan is not None and nbytes is None) else (nbytes or 0)
        return L.mla_decode_forward_step(ctypes.byref(plan) if plan is not None else None,
                                         ctypes.byref(args) if args is not None else None,
                                         ctypes.c_void_p(scratch) if scratch else None, nb, new_rows, adv, None)

    assert call(None, a, rows, 1) == mla.EINVAL
    assert call(p, a, None, 1) == mla.EINVAL
    assert call(p, a, rows, 2) == mla.EINVAL
    assert call(p, a, rows, -1) == mla.EINVAL
    assert call(p, a, ctypes.c_void_p(0x70008), 1) == mla.EALIGN
    assert call(p, None, rows, 0) == mla.EINVAL
    assert call(p, a, rows, 1, scratch=0) == mla.ESCRATCH
    assert call(p, a, rows, 1, nbytes=16) == mla.ESCRATCH
    ps = _plan(sparse=True, topk=64)
    assert call(ps, _args(row_offset=0x60000, indices=0x61000, cache_len=0x62000), rows, 1) == mla.EUNSUPPORTED
    bad = mla.Plan.from_buffer_copy(p)
    bad.magic = 0
    assert call(bad, a, rows, 1) == mla.EINVAL


def test_fp8_cache_plan_and_argument_checks():
    """E4M3 caches: dense on the warp-MMA kernel only (P . V on the warps or on
    tcgen05); the scale and the byte row stride are checked before any launch."""
    p = _plan(max_ctx=4096, kv_fp8=True)
    assert p.variant == 5 and p.shape.kv_fp8 == 1            # automatic: P . V on tcgen05
    assert 0 < p.smem_bytes <= 227 * 1024
    assert _plan(heads=128, max_ctx=131072, kv_fp8=True).variant == 5   # the warp-MMA kernel at any width
    assert _plan(max_ctx=4096, kv_fp8=True, variant=1).variant == 1
    L = mla.lib()
    s = mla.Shape(batch=1, heads=16, d_latent=512, d_rope=64, sparse=0, max_ctx=64, topk=0, scale=SCALE,
                  num_sms=152, splits_override=0, variant=0, pdl=0, stall_test=0, kv_fp8=2)
    out = mla.Plan()
    assert L.mla_decode_plan(ctypes.byref(s), ctypes.byref(out)) == mla.EINVAL
    for kw, rc in [(dict(sparse=1, topk=64), mla.EUNSUPPORTED), (dict(variant=2), mla.EUNSUPPORTED),
                   (dict(variant=4, heads=64), mla.EUNSUPPORTED)]:
        s = mla.Shape(batch=1, heads=kw.get("heads", 16), d_latent=512, d_rope=64, sparse=kw.get("sparse", 0),
                      max_ctx=64, topk=kw.get("topk", 0), scale=SCALE, num_sms=152, splits_override=0,
                      variant=kw.get("variant", 0), pdl=0, stall_test=0, kv_fp8=1)
        assert L.mla_decode_plan(ctypes.byref(s), ctypes.byref(out)) == rc, kw
    for a, rc in [(_args(kv_scale=0.0), mla.EINVAL), (_args(kv_scale=float("nan")), mla.EINVAL),
                  (_args(kv_scale=-1.0), mla.EINVAL), (_args(kv_scale=float("inf")), mla.EINVAL),
                  (_args(kv_scale=0.5, row_stride=584), mla.EALIGN)]:
        for fn in ("mla_decode_run", "mla_decode_combine", "mla_decode_forward"):
            assert _call(fn, p, a) == rc, (fn, a.kv_scale, a.row_stride)
    rows = ctypes.c_void_p(0x70000)
    assert L.mla_decode_forward_step(ctypes.byref(p), ctypes.byref(_args(kv_scale=1.0)), ctypes.c_void_p(0x100000),
                                     p.scratch_bytes, rows, 1, None) == mla.EUNSUPPORTED


def test_plan_warp_mma_with_tcgen05_pv():
    """Variant 5 (scores on the warps, P . V on tcgen05) plans like the warp-MMA
    kernel: 16 heads per CTA, 32-row granule and modelled step, the same split
    rule; dense caches (bf16 or E4M3) only."""
    for T in (256, 8192, 131072):
        a = _plan(max_ctx=T, variant=1)
        b = _plan(max_ctx=T, variant=5)
        assert b.variant == 5 and b.head_group == 16 and b.block == a.block
        assert (b.splits, b.entries_per_split, b.grid_x, b.combine_grid_x) == \
            (a.splits, a.entries_per_split, a.grid_x, a.combine_grid_x)
        assert b.scratch_bytes == a.scratch_bytes
    assert _plan(max_ctx=8192, heads=64, variant=5).n_head_groups == 4
    f = _plan(max_ctx=8192, variant=5, kv_fp8=True)
    assert f.variant == 5 and f.shape.kv_fp8 == 1 and 0 < f.smem_bytes <= 227 * 1024
    with pytest.raises(mla.MLADecodeError) as e:
        _plan(sparse=True, topk=64, variant=5, kv_fp8=True)
    assert e.value.status == mla.EUNSUPPORTED



def test_floor_probes_reject_bad_arguments():
    """The floor probes check every argument before anything is launched."""
    L = mla.lib()
    pair = L.mla_floor_empty_pair
    ok = (128, 384, 200000)
    assert pair(*ok, *ok, 2, None) == mla.EINVAL
    for bad in ((0, 384, 0), (65536, 384, 0), (128, 16, 0), (128, 33, 0), (128, 2048, 0), (128, 384, -1),
                (128, 384, 227 * 1024 + 1)):
        assert pair(*bad, *ok, 1, None) == mla.EINVAL, bad
        assert pair(*ok, *bad, 1, None) == mla.EINVAL, bad
    read = L.mla_floor_read
    p16 = ctypes.c_void_p(0x10000)
    assert read(None, 4096, 8, p16, p16, 1, None) == mla.EINVAL
    assert read(p16, 0, 8, p16, p16, 1, None) == mla.EINVAL
    assert read(p16, 4096, 0, p16, p16, 1, None) == mla.EINVAL
    assert read(p16, 4096, 65536, p16, p16, 1, None) == mla.EINVAL
    assert read(p16, 4096, 8, None, p16, 1, None) == mla.EINVAL
    assert read(p16, 4096, 8, p16, None, 1, None) == mla.EINVAL
    assert read(p16, 4096, 8, p16, p16, 3, None) == mla.EINVAL
    assert read(p16, 4100, 8, p16, p16, 1, None) == mla.EALIGN
    assert read(ctypes.c_void_p(0x10008), 4096, 8, p16, p16, 1, None) == mla.EALIGN
    assert read(p16, 4096, 8, ctypes.c_void_p(0x10002), p16, 1, None) == mla.EALIGN
    assert read(p16, 4096, 8, p16, ctypes.c_void_p(0x10001), 1, None) == mla.EALIGN


def test_floor_gather_rejects_bad_arguments():
    g = mla.lib().mla_floor_gather
    p16, p8 = ctypes.c_void_p(0x10000), ctypes.c_void_p(0x10008)
    ok = dict(kv=p16, kv_rows=100, row_stride=1152, row_bytes=1152, rows=p8, n_rows=10, ctas=4, sink=p16,
              status=p16, pdl=1)

    def call(**kw):
        a = dict(ok)
        a.update(kw)
        return g(a["kv"], a["kv_rows"], a["row_stride"], a["row_bytes"], a["rows"], a["n_rows"], a["ctas"],
                 a["sink"], a["status"], a["pdl"], None)

    for bad in (dict(kv=None), dict(rows=None), dict(sink=None), dict(status=None), dict(kv_rows=0),
                dict(n_rows=0), dict(ctas=0), dict(ctas=65536), dict(row_bytes=0), dict(row_bytes=98320),
                dict(row_stride=1136), dict(pdl=2)):
        assert call(**bad) == mla.EINVAL, bad
    for bad in (dict(row_bytes=1160, row_stride=1168), dict(row_stride=1160), dict(kv=p8),
                dict(rows=ctypes.c_void_p(0x10004)), dict(sink=ctypes.c_void_p(0x10002)),
                dict(status=ctypes.c_void_p(0x10001))):
        assert call(**bad) == mla.EALIGN, bad
