"""C-ABI checks that need no GPU: libfd.so loads, exports every entry point
include/fd_decode_attn.h declares, plans as documented, and rejects bad
arguments before making any CUDA call."""

import ctypes
import re
from pathlib import Path

import pytest

import decode_attention_04_gb300 as fd
from decode_attention_04_gb300.inputs import WORKLOADS

ROOT = Path(__file__).resolve().parent.parent


@pytest.fixture(scope="module")
def lib():
    from decode_attention_04_gb300 import build
    build.build()
    return fd.load_library()


def _declared():
    names = set()
    for h in (ROOT / "include").glob("*.h"):
        text = re.sub(r"/\*.*?\*/", "", h.read_text(), flags=re.S)
        names |= set(re.findall(r"\b(fd_\w+)\s*\(", text))
    return names


def test_header_declares_the_boundary():
    d = _declared()
    for n in ("fd_plan", "fd_decode_attn", "fd_decode_attn_ex", "fd_strerror", "fd_get_device_error"):
        assert n in d


def test_every_declared_symbol_is_exported(lib):
    missing = [n for n in sorted(_declared()) if not hasattr(lib, n)]
    assert not missing, missing
    # the binding wraps every one of them under the same name
    for n in _declared():
        assert callable(getattr(fd, n)), n


def test_strerror_and_version(lib):
    assert fd.fd_strerror(fd.FD_OK) == "ok"
    for c in (1, 2, 3, 4, 5):
        assert fd.fd_strerror(c) and fd.fd_strerror(c) != "unknown status"
    assert fd.fd_strerror(99) == "unknown status"
    assert fd.fd_version() > 0


def _plan(w, sms=152, ctas=2, max_len=0):
    return fd.fd_plan_sms(w.B, w.NH, w.NKV, w.HS, w.capacity, w.window, max_len, sms, ctas)


@pytest.mark.parametrize("name", sorted(WORKLOADS))
def test_plan_fills_the_gpu_and_sizes_workspace(name, lib):
    w = WORKLOADS[name]
    p = _plan(w)
    units = w.B * w.NKV
    band = min(w.window if w.window > 0 else w.capacity, w.capacity)
    assert p.max_band == band
    # every CTA slot of the GPU gets work at the bound the plan was sized for
    chunk = -(-band // p.num_splits)
    chunk = -(-chunk // p.granule) * p.granule
    active = -(-band // chunk)
    # one block per CTA slot (per SM when G >= 8, where partials are costly)
    per_sm = 1 if w.G >= 8 else 2
    assert units * active >= 0.9 * min(152 * per_sm, units * -(-band // p.granule))
    P = p.num_splits // p.cluster
    assert p.num_splits % p.cluster == 0
    up = lambda x: -(-x // 256) * 256
    expect_zero = 0 if P == 1 else up(w.B * w.NKV * 4)
    expect_ws = 0 if P == 1 else expect_zero + up(w.B * w.NH * P * w.HS * 4) + up(w.B * w.NH * P * 8)
    assert p.workspace_zero_bytes == expect_zero
    assert p.fused == 0  # the fused merge is opt-in
    G = w.NH // w.NKV
    if P > 1 and G * p.num_splits * w.HS * 4 <= 256 << 10:
        q = fd.fd_plan_t.from_buffer_copy(p)
        fd.fd_plan_override(q, 0, 0, 0, 1)
        assert q.fused == 1 and q.workspace_bytes == p.workspace_bytes
    assert p.workspace_bytes == expect_ws == fd.fd_workspace_bytes(p)
    # workspace is bounded by partials, never by the cache allocation
    assert p.workspace_bytes <= 32 << 20


def test_plan_mqa_one_kv_head_uses_every_sm(lib):
    w = WORKLOADS["gemma_global_mqa_32k"]
    p = _plan(w)
    assert p.num_splits >= 152  # one KV head still spreads over all SMs
    assert p.cluster == 1  # clusters are opt-in


def test_plan_uses_no_clusters_by_default(lib):
    for name in WORKLOADS:
        assert _plan(WORKLOADS[name]).cluster == 1


def test_plan_max_len_tightens_short_context(lib):
    w = WORKLOADS["gemma_global_mqa_4k"]
    full = _plan(w)
    short = _plan(w, max_len=4096)
    assert short.max_band == 4096 < full.max_band
    assert short.workspace_bytes <= full.workspace_bytes


def test_plan_balance_bound_for_ragged_batches(lib):
    w = WORKLOADS["llama_ragged"]
    p = _plan(w)
    chunk = -(-w.capacity // p.num_splits)
    assert chunk * w.HS * 4 <= (2 << 20) + p.granule * w.HS * 4
    assert p.num_splits % max(1, -(-(152 * 2) // (w.B * w.NKV))) == 0  # whole waves


def test_plan_override(lib):
    w = WORKLOADS["gemma_local_ring"]
    p = _plan(w)
    fd.fd_plan_override(p, 1, fd.FD_PATH_SIMT)
    assert p.num_splits == 1 and p.path == fd.FD_PATH_SIMT and p.workspace_bytes == 0
    fd.fd_plan_override(p, 7, fd.FD_PATH_TC)
    assert p.num_splits == 7 and p.path == fd.FD_PATH_TC and p.workspace_bytes > 0
    with pytest.raises(fd.FdError):
        fd.fd_plan_override(p, -1, 0)
    with pytest.raises(fd.FdError):
        fd.fd_plan_override(p, 0, 9)
    # clusters: powers of two <= 16 dividing S (and HS / 4); tensor-core path only
    fd.fd_plan_override(p, 32, fd.FD_PATH_TC, 8)
    assert p.cluster == 8 and p.workspace_bytes == fd.fd_workspace_bytes(p) > 0
    fd.fd_plan_override(p, 16, 0, 16)
    assert p.cluster == 16 and p.workspace_bytes == 0  # one cluster spans every split
    for bad in [(24, 0, 16), (32, 0, 3), (32, 0, 32), (32, fd.FD_PATH_SIMT, 8)]:
        q = fd.fd_plan_t.from_buffer_copy(p)
        with pytest.raises(fd.FdError):
            fd.fd_plan_override(q, *bad)
    fd.fd_plan_override(p, 5, fd.FD_PATH_SIMT, 1)
    assert p.cluster == 1 and p.path == fd.FD_PATH_SIMT


@pytest.mark.parametrize("args,code", [
    ((1, 16, 8, 96, 64, 0), fd.FD_ERR_UNSUPPORTED),     # HS
    ((1, 12, 8, 128, 64, 0), fd.FD_ERR_UNSUPPORTED),    # NH % NKV
    ((1, 64, 2, 128, 64, 0), fd.FD_ERR_UNSUPPORTED),    # G = 32 > 16
    ((1, 16, 8, 128, 64, 65), fd.FD_ERR_INVALID_ARG),   # window > capacity
    ((1, 16, 8, 128, 0, 0), fd.FD_ERR_INVALID_ARG),     # capacity
    ((-1, 16, 8, 128, 64, 0), fd.FD_ERR_INVALID_ARG),   # B
    ((1, 0, 8, 128, 64, 0), fd.FD_ERR_INVALID_ARG),     # NH
])
def test_shape_errors_before_any_cuda_call(lib, args, code):
    B, NH, NKV, HS, cap, win = args
    p = fd.fd_plan_t()
    assert lib.fd_plan_sms(B, NH, NKV, HS, cap, win, 0, 152, 2, 8, ctypes.byref(p)) == code
    # fd_decode_attn checks the shape before it touches the device
    assert lib.fd_decode_attn(16, 16, 16, 16, 16, B, NH, NKV, HS, cap, win, 0.0, None) == code


def test_pointer_and_workspace_errors_before_any_cuda_call(lib):
    w = WORKLOADS["gemma_local_ring"]
    p = _plan(w)
    args = (w.B, w.NH, w.NKV, w.HS, w.capacity, w.window, 0.0, None)
    A = 1 << 20  # fake, aligned addresses; nothing is dereferenced on these paths
    ex = lib.fd_decode_attn_ex
    # null tensor
    assert ex(ctypes.byref(p), A, p.workspace_bytes, None, None, A, A, A, A, *args) == fd.FD_ERR_INVALID_ARG
    # misaligned q / lens / out_f32
    assert ex(ctypes.byref(p), A, p.workspace_bytes, None, A + 2, A, A, A, A, *args) == fd.FD_ERR_ALIGNMENT
    assert ex(ctypes.byref(p), A, p.workspace_bytes, None, A, A, A, A, A + 2, *args) == fd.FD_ERR_ALIGNMENT
    assert ex(ctypes.byref(p), A, p.workspace_bytes, A + 4, A, A, A, A, A, *args) == fd.FD_ERR_ALIGNMENT
    # workspace missing / too small / misaligned
    assert ex(ctypes.byref(p), None, 0, None, A, A, A, A, A, *args) == fd.FD_ERR_WORKSPACE
    assert ex(ctypes.byref(p), A, p.workspace_bytes - 1, None, A, A, A, A, A, *args) == fd.FD_ERR_WORKSPACE
    assert ex(ctypes.byref(p), A + 8, p.workspace_bytes, None, A, A, A, A, A, *args) == fd.FD_ERR_ALIGNMENT
    # shape that disagrees with the plan
    bad = (w.B, w.NH, w.NKV, w.HS, w.capacity * 2, w.window, 0.0, None)
    assert ex(ctypes.byref(p), A, p.workspace_bytes, None, A, A, A, A, A, *bad) == fd.FD_ERR_INVALID_ARG
    # null plan
    assert ex(None, A, p.workspace_bytes, None, A, A, A, A, A, *args) == fd.FD_ERR_INVALID_ARG
    # B == 0 is a no-op success
    p0 = fd.fd_plan_sms(0, 16, 8, 256, 64, 0, 0, 152, 2, 8)
    assert ex(ctypes.byref(p0), None, 0, None, None, None, None, None, None,
              0, 16, 8, 256, 64, 0, 0.0, None) == fd.FD_OK
    assert lib.fd_get_device_error(None, None) == fd.FD_ERR_INVALID_ARG


def test_binding_raises_fderror(lib):
    with pytest.raises(fd.FdError) as e:
        fd.fd_plan_sms(1, 16, 8, 96, 64, 0, 0, 152, 2)
    assert e.value.status == fd.FD_ERR_UNSUPPORTED


def _plan_kv(w, kv=fd.FD_KV_E4M3, sms=152, ctas=2, max_len=0):
    return fd.fd_plan_sms_kv(w.B, w.NH, w.NKV, w.HS, w.capacity, w.window, max_len, sms, ctas, 8, kv)


@pytest.mark.parametrize("name", sorted(WORKLOADS))
def test_e4m3_plan_matches_bf16_rule_with_half_the_bytes(name, lib):
    w = WORKLOADS[name]
    p8, p16 = _plan_kv(w), _plan(w)
    assert p8.kv_dtype == fd.FD_KV_E4M3 and p16.kv_dtype == fd.FD_KV_BF16
    # 1 KB E4M3 groups for head dim 256 with more than 8 query rows, and for
    # 64 / 128 when the band is cut into whole short tiles (the half-length
    # tile: 64 positions at d128)
    short = w.HS in (64, 128) and p8.granule > 1
    assert p8.group_bytes == (1024 if (w.HS == 256 and w.G > 8) or short else 2048) and p8.path == fd.FD_PATH_TC
    if short:
        assert p8.granule == {64: 128, 128: 64}[w.HS]
    # consumer warps: 8 for the E4M3 head-dim-512 MQA tile only when the grid
    # is one block per SM; bf16 head dims 256/512 (16-row tiles) use 8
    blocks = w.B * w.NKV * p8.num_splits
    if w.HS == 512 and w.G > 8:
        assert p8.consumer_warps == (8 if blocks <= 152 else 4)
    assert p16.consumer_warps == (8 if w.HS == 256 or (w.HS == 512 and w.G > 8) else 4)
    # the same SM fill; a split is bounded by the same ~2 MiB of K+V bytes,
    # which at 2 bytes per position pair is twice the positions
    chunk8 = -(-p8.max_band // p8.num_splits)
    assert chunk8 * w.HS * 2 <= (2 << 20) + w.HS * 2
    if p8.granule == p16.granule:  # whole-tile splits of different tile lengths differ in count
        assert p8.num_splits <= p16.num_splits
    # a bf16 plan from fd_plan_sms_kv is fd_plan_sms's plan
    same = _plan_kv(w, fd.FD_KV_BF16)
    assert bytes(same) == bytes(p16)


def test_e4m3_plan_rejects_the_simt_path_and_unknown_types(lib):
    w = WORKLOADS["gemma_local_ring"]
    p = _plan_kv(w)
    with pytest.raises(fd.FdError) as e:
        fd.fd_plan_override(p, 0, fd.FD_PATH_SIMT)
    assert e.value.status == fd.FD_ERR_INVALID_ARG
    fd.fd_plan_override(p, 9, fd.FD_PATH_TC)  # split count and clusters still move
    assert p.num_splits == 9 and p.group_bytes == 2048 and p.consumer_warps == 8
    # the E4M3 MQA tile follows the grid: one block per SM -> 8 warps, more -> 4
    m = _plan_kv(WORKLOADS["gemma_global_mqa_32k"])
    assert m.num_splits * m.B * m.NKV <= 152 and m.consumer_warps == 8
    fd.fd_plan_override(m, 2 * m.num_splits)
    assert m.consumer_warps == 4
    pp = fd.fd_plan_t()
    assert lib.fd_plan_sms_kv(1, 16, 8, 256, 64, 0, 0, 152, 2, 8, 2, ctypes.byref(pp)) == fd.FD_ERR_INVALID_ARG
    assert lib.fd_plan_kv(1, 16, 8, 256, 64, 0, 0, 0, 7, ctypes.byref(pp)) == fd.FD_ERR_INVALID_ARG


def test_e4m3_argument_errors_before_any_cuda_call(lib):
    w = WORKLOADS["gemma_local_ring"]
    p8, p16 = _plan_kv(w), _plan(w)
    args = (w.B, w.NH, w.NKV, w.HS, w.capacity, w.window, 0.0, None)
    A = 1 << 20  # fake, aligned addresses; nothing is dereferenced on these paths
    ex8, ex16 = lib.fd_decode_attn_fp8_ex, lib.fd_decode_attn_ex
    ws = p8.workspace_bytes
    # a plan of the other cache type
    assert ex8(ctypes.byref(p16), A, p16.workspace_bytes, None, A, A, A, A, A, A, A, *args) == fd.FD_ERR_INVALID_ARG
    assert ex16(ctypes.byref(p8), A, ws, None, A, A, A, A, A, *args) == fd.FD_ERR_INVALID_ARG
    # missing or misaligned scales
    assert ex8(ctypes.byref(p8), A, ws, None, A, A, A, None, A, A, A, *args) == fd.FD_ERR_INVALID_ARG
    assert ex8(ctypes.byref(p8), A, ws, None, A, A, A, A, None, A, A, *args) == fd.FD_ERR_INVALID_ARG
    assert ex8(ctypes.byref(p8), A, ws, None, A, A, A, A + 2, A, A, A, *args) == fd.FD_ERR_ALIGNMENT
    # misaligned codes, short workspace
    assert ex8(ctypes.byref(p8), A, ws, None, A, A + 8, A, A, A, A, A, *args) == fd.FD_ERR_ALIGNMENT
    assert ex8(ctypes.byref(p8), A, ws - 1, None, A, A, A, A, A, A, A, *args) == fd.FD_ERR_WORKSPACE
    # the auto entry point checks shapes and scales before touching the device
    bad = (1, 16, 8, 96, 64, 0, 0.0, None)
    assert lib.fd_decode_attn_fp8(A, A, A, A, A, A, A, *bad) == fd.FD_ERR_UNSUPPORTED
    assert lib.fd_decode_attn_fp8(A, A, A, None, A, A, A, *args) == fd.FD_ERR_INVALID_ARG


def test_short_bands_split_into_whole_tiles(lib):
    """Where filling the GPU would cut the band into pieces under two tiles,
    the chunk granule is the tile (64 positions at d128, and at d256 for up to
    8 query rows: the sliding ring's tile copies 4 KB groups), so a split is
    never a sliver of a tile; long bands keep granule 1."""
    tiny, ring = _plan(WORKLOADS["llama_tiny"]), _plan(WORKLOADS["gemma_local_ring"])
    assert tiny.granule == 64 and ring.granule == 64
    for p in (tiny, ring):
        chunk = -(-p.max_band // p.num_splits)
        chunk = -(-chunk // p.granule) * p.granule
        assert chunk % p.granule == 0 and chunk >= p.granule
    assert ring.num_splits == 16  # 1024 / 64: one tile per split
    for name in ("gemma_global_mqa_32k", "llama_ragged", "gemma_mqa_long"):
        assert _plan(WORKLOADS[name]).granule == 1
    # a forced split count keeps the plan's granule; a forced family resets it
    p = _plan(WORKLOADS["llama_tiny"])
    fd.fd_plan_override(p, 3)
    assert p.granule == 64
    fd.fd_plan_override(p, 0, fd.FD_PATH_SIMT)
    assert p.granule == 1


def test_tcgen05_family_is_opt_in_and_shape_bound(lib):
    """Plans never pick FD_PATH_UMMA; it is accepted for bf16, head dim 512,
    8 < G <= 16 and no window, with its own copy-group and warp fields."""
    for name in WORKLOADS:
        assert _plan(WORKLOADS[name]).path == fd.FD_PATH_TC
    p = _plan(WORKLOADS["gemma_global_mqa_32k"])
    fd.fd_plan_override(p, 0, fd.FD_PATH_UMMA)
    assert p.path == fd.FD_PATH_UMMA and p.group_bytes == 16384 and p.consumer_warps == 4
    assert p.granule == 16  # only the band's last split can end off a 16-row P.V step
    for w in (WORKLOADS["gemma_local_ring"], WORKLOADS["llama_tiny"]):
        q = _plan(w)
        with pytest.raises(fd.FdError):
            fd.fd_plan_override(q, 0, fd.FD_PATH_UMMA)
    e = _plan_kv(WORKLOADS["gemma_global_mqa_32k"])
    with pytest.raises(fd.FdError):
        fd.fd_plan_override(e, 0, fd.FD_PATH_UMMA)  # bf16 only
    for bad in [(0, fd.FD_PATH_UMMA, 2), (0, fd.FD_PATH_UMMA, 0, 1)]:
        q = fd.fd_plan_t.from_buffer_copy(p)
        with pytest.raises(fd.FdError):
            fd.fd_plan_override(q, *bad)


def test_persistent_grid_is_opt_in_and_sized(lib):
    """fd_plan_persistent: one block per resident slot (or per item), one more
    zeroed counter word in the workspace, tensor-core path without clusters or
    the fused merge only; fd_plan_override returns to the plan's rule."""
    up = lambda x: -(-x // 256) * 256
    for name in WORKLOADS:
        assert _plan(WORKLOADS[name]).persistent == 0
    w = WORKLOADS["llama_ragged"]
    p = _plan(w)
    items = p.num_splits * w.NKV * w.B
    q = fd.fd_plan_t.from_buffer_copy(p)
    fd.fd_plan_persistent(q, 1)
    assert q.persistent == min(items, 152 * 2)
    assert q.workspace_zero_bytes == up((w.B * w.NKV + 1) * 4)
    assert q.workspace_bytes == p.workspace_bytes - p.workspace_zero_bytes + q.workspace_zero_bytes
    assert q.workspace_bytes == fd.fd_workspace_bytes(q)
    assert (q.num_splits, q.group_bytes, q.consumer_warps) == (p.num_splits, p.group_bytes, p.consumer_warps)
    fd.fd_plan_persistent(q, 0)
    assert q.persistent == 0 and q.workspace_bytes == p.workspace_bytes
    # fewer items than block slots: one block per item; S = 1 still needs the counter
    t = WORKLOADS["llama_tiny"]
    s1 = _plan(t)
    fd.fd_plan_override(s1, 1)
    assert s1.workspace_bytes == 0
    fd.fd_plan_persistent(s1, 1)
    assert s1.persistent == t.B * t.NKV and s1.workspace_bytes == s1.workspace_zero_bytes == 256
    fd.fd_plan_override(s1, 2)
    assert s1.persistent == 0  # back to the plan's rule
    # not available: SIMT path, clusters, fused merge; bad modes
    for args in [(0, fd.FD_PATH_SIMT, 0, -1), (32, fd.FD_PATH_TC, 2, -1), (0, 0, 0, 1)]:
        r = _plan(WORKLOADS["gemma_local_ring"])
        fd.fd_plan_override(r, *args)
        with pytest.raises(fd.FdError):
            fd.fd_plan_persistent(r, 1)
        fd.fd_plan_persistent(r, 0)
        fd.fd_plan_persistent(r, -1)
        assert r.persistent == 0
    for mode in (2, -2):
        with pytest.raises(fd.FdError):
            fd.fd_plan_persistent(fd.fd_plan_t.from_buffer_copy(p), mode)


def test_persistent_plan_checked_before_any_cuda_call(lib):
    """A persistent plan with a block count outside [1, items], or one whose
    path cannot run it, is refused by fd_decode_attn_ex before any launch."""
    w = WORKLOADS["llama_tiny"]
    p = _plan(w)
    fd.fd_plan_persistent(p, 1)
    items = p.num_splits * w.NKV * w.B
    dummy = ctypes.c_void_p(256)  # never dereferenced: the plan check comes first
    for bad in (-1, items + 1):
        q = fd.fd_plan_t.from_buffer_copy(p)
        q.persistent = bad
        rc = lib.fd_decode_attn_ex(ctypes.byref(q), dummy, q.workspace_bytes, None, dummy, dummy, dummy, dummy,
                                   dummy, w.B, w.NH, w.NKV, w.HS, w.capacity, w.window, 0.0, None)
        assert rc == fd.FD_ERR_INVALID_ARG
    q = fd.fd_plan_t.from_buffer_copy(p)
    q.path, q.consumer_warps = fd.FD_PATH_SIMT, 0  # a valid SIMT plan but for the persistent grid
    rc = lib.fd_decode_attn_ex(ctypes.byref(q), dummy, q.workspace_bytes, None, dummy, dummy, dummy, dummy,
                               dummy, w.B, w.NH, w.NKV, w.HS, w.capacity, w.window, 0.0, None)
    assert rc == fd.FD_ERR_INVALID_ARG


def test_e4m3_short_band_tile(lib):
    """An E4M3 cache with head dim 128 and a short band takes the half-length
    tile (1 KB groups, 64 positions): twice the splits of the 2 KB tile; long
    bands keep 2 KB groups; a forced kernel family returns to the default."""
    t = WORKLOADS["llama_tiny"]
    p = _plan_kv(t)
    assert (p.granule, p.group_bytes) == (64, 1024)
    assert p.num_splits == -(-t.capacity // 64)
    r = _plan_kv(WORKLOADS["llama_ragged"])
    assert (r.granule, r.group_bytes) == (1, 2048)
    fd.fd_plan_override(p, 0, fd.FD_PATH_TC)  # same family: unchanged
    assert p.group_bytes == 1024
    q = _plan_kv(WORKLOADS["gemma_local_ring"])
    assert q.group_bytes == 2048 and q.granule == 64  # the ring's tile: 2 KB E4M3 groups, 64 positions


def test_compiled_entries_return_the_library_status(lib):
    """The compiled CPython entries (built where Python headers exist) call
    the same loaded libfd.so as ctypes: argument errors come back as the same
    status codes, before any CUDA call."""
    f = fd._fast()
    if f is None:
        pytest.skip("compiled entries not built here")
    cases = [(0, 0, 0, 0, 0, 1, 16, 8, 256, 64, 0, 0.0, 0),          # null pointers
             (16, 16, 16, 16, 16, 1, 16, 8, 96, 64, 0, 0.0, 0),      # unsupported head size
             (16, 16, 16, 16, 16, 1, 16, 8, 256, 64, 65, 0.0, 0)]    # window > capacity
    for c in cases:
        assert f.decode_attn(*c) == lib.fd_decode_attn(*c) != fd.FD_OK
    c8 = (0, 0, 0, 0, 0, 0, 0, 1, 16, 8, 256, 64, 0, 0.0, 0)
    assert f.decode_attn_fp8(*c8) == lib.fd_decode_attn_fp8(*c8) == fd.FD_ERR_INVALID_ARG
    # explicit-plan entries: a null plan, and a plan made for another shape
    tail = (16, 16, 16, 16, 16, 1, 16, 8, 256, 64, 0, 0.0, 0)
    assert f.decode_attn_ex(0, 0, 0, 0, *tail) == lib.fd_decode_attn_ex(None, None, 0, None, *tail) \
        == fd.FD_ERR_INVALID_ARG
    other = _plan(WORKLOADS["llama_tiny"])
    assert f.decode_attn_ex(ctypes.addressof(other), 0, 0, 0, *tail) == \
        lib.fd_decode_attn_ex(ctypes.byref(other), None, 0, None, *tail) == fd.FD_ERR_INVALID_ARG
    tail8 = (16, 16, 16, 16, 16, 16, 16, 1, 16, 8, 256, 64, 0, 0.0, 0)
    assert f.decode_attn_fp8_ex(0, 0, 0, 0, *tail8) == lib.fd_decode_attn_fp8_ex(None, None, 0, None, *tail8) \
        == fd.FD_ERR_INVALID_ARG


def test_plan_long_bands_with_large_groups_fill_every_slot_once(lib):
    """G >= 8: one block per SM while a split stays under ~2 MiB of K+V; a
    longer band (MQA, 4 x 131072 positions) first takes every resident slot
    once with up to ~4 MiB per split; B = 1 MQA at 32K keeps one per SM."""
    w = WORKLOADS["gemma_mqa_long"]
    p = _plan(w)
    assert w.G >= 8 and p.num_splits * w.B * w.NKV == 152 * 2
    assert -(-w.capacity // p.num_splits) * w.HS * 4 <= 4 << 20
    assert _plan(WORKLOADS["gemma_global_mqa_32k"]).num_splits == 152
    one_per_sm = _plan(w, ctas=1)  # no second slot per SM: waves at the 2 MiB bound
    assert -(-w.capacity // one_per_sm.num_splits) * w.HS * 4 <= (2 << 20) + w.HS * 4


def test_plan_min_len_recorded_and_checked(lib):
    """fd_plan_min_len records the caller's lower bound on the lengths; plans
    start with none; a negative bound is refused; overrides keep it."""
    w = WORKLOADS["gemma_local_ring"]
    p = _plan(w)
    assert p.min_len == 0
    fd.fd_plan_min_len(p, w.capacity)
    assert p.min_len == w.capacity
    fd.fd_plan_override(p, 7, 0, 0, -1)
    assert p.min_len == w.capacity and p.num_splits == 7
    assert lib.fd_plan_min_len(ctypes.byref(p), -1) == fd.FD_ERR_INVALID_ARG
    assert lib.fd_plan_min_len(None, 5) == fd.FD_ERR_INVALID_ARG
    assert p.min_len == w.capacity


def test_group_step_plan_rules(lib):
    """fused = 2 (the group step): allowed on the tensor-core path without
    clusters when the whole grid is resident at once (B * NKV * S <= SMs x
    CTAs per SM); the counter region doubles (count-in and count-out words,
    both zeroed); refused beyond one wave, with clusters, with the persistent
    grid, and for fused values other than -1..2."""
    up = lambda x: -(-x // 256) * 256
    w = WORKLOADS["gemma_local_ring"]
    p = _plan(w)  # 152 SMs x 2 CTAs
    q = fd.fd_plan_t.from_buffer_copy(p)
    fd.fd_plan_override(q, 0, 0, 0, 2)
    assert q.fused == 2 and q.num_splits == p.num_splits
    assert q.workspace_zero_bytes == up(2 * w.B * w.NKV * 4)
    assert q.workspace_bytes == p.workspace_bytes - p.workspace_zero_bytes + q.workspace_zero_bytes
    assert q.workspace_bytes == fd.fd_workspace_bytes(q)
    cap = 152 * 2 // (w.B * w.NKV)
    fd.fd_plan_override(q, cap, 0, 0, 2)
    assert q.fused == 2
    for args in [(cap + 1, 0, 1, 2), (32, 0, 2, 2), (0, fd.FD_PATH_SIMT, 0, 2), (0, 0, 0, 3)]:
        with pytest.raises(fd.FdError):
            fd.fd_plan_override(fd.fd_plan_t.from_buffer_copy(p), *args)
    with pytest.raises(fd.FdError):
        fd.fd_plan_persistent(q, 1)
    fd.fd_plan_override(q, 0, 0, 0, 0)
    assert q.fused == 0 and q.workspace_bytes == fd.fd_workspace_bytes(q)
    # a hand-edited plan with an unknown mode is refused before any launch
    bad = fd.fd_plan_t.from_buffer_copy(p)
    bad.fused = 3
    dummy = ctypes.c_void_p(256)
    rc = lib.fd_decode_attn_ex(ctypes.byref(bad), dummy, bad.workspace_bytes, None, dummy, dummy, dummy, dummy,
                               dummy, w.B, w.NH, w.NKV, w.HS, w.capacity, w.window, 0.0, None)
    assert rc == fd.FD_ERR_INVALID_ARG


# (workload) -> (bf16 splits, granule, group bytes), (E4M3 splits, granule, group bytes)
# on 152 SMs x 2 CTAs: the sliding ring takes 64-position tiles (4 KB bf16 / 2 KB
# E4M3 groups) as 16 one-tile splits; B = 1 MQA the wide 4 KB tile; Llama tiny
# whole 64-position tiles (the E4M3 half-length 1 KB tile)
PLAN_TABLE = {
    "llama_tiny": ((8, 64, 2048), (8, 64, 1024)),
    "gemma_local_ring": ((16, 64, 4096), (16, 64, 2048)),
    "gemma_global_mqa_4k": ((152, 1, 4096), (152, 1, 2048)),
    "gemma_global_mqa_32k": ((152, 1, 4096), (152, 1, 2048)),
    "llama_ragged": ((9, 1, 2048), (6, 1, 2048)),
    "gemma_mqa_long": ((76, 1, 2048), (76, 1, 2048)),
}


@pytest.mark.parametrize("name", sorted(PLAN_TABLE))
def test_plan_table_of_the_benchmark_workloads(name, lib):
    """The split count, chunk granule and copy-group size each benchmark
    workload's plan takes, for both cache types."""
    w = WORKLOADS[name]
    p, p8 = _plan(w), _plan_kv(w)
    want, want8 = PLAN_TABLE[name]
    assert (p.num_splits, p.granule, p.group_bytes) == want
    assert (p8.num_splits, p8.granule, p8.group_bytes) == want8
