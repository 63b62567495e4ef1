"""Host-side checks of the C ABI (no GPU): the library loads, exports every entry point
include/gdn.h declares, and rejects bad arguments before launching anything.

The rejection tests hand the library fake device addresses; they only run where no CUDA
device exists (validation must return first, so nothing is ever dereferenced there).
"""
import ctypes
import os
import re

import pytest
import torch

from gated_deltanet_linear_11_gb300 import _lib, build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "gdn.h")


@pytest.fixture(scope="module")
def lib():
    build.build()
    return _lib.load()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(gdn_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for want in ("gdn_conv1d_fwd", "gdn_conv1d_update", "gdn_chunk_prefill",
                 "gdn_recurrent_decode", "gdn_chunk_prefill_workspace_size",
                 "gdn_status_string", "gdn_version"):
        assert want in names


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name
    assert set(_lib.EXPORTS) <= set(declared_functions())


def test_status_strings_and_version(lib):
    assert lib.gdn_version() >= 100
    for code, name in _lib.STATUS.items():
        assert lib.gdn_status_string(code).decode().startswith(name)


def test_missing_library_fails_loudly(tmp_path):
    saved = _lib._lib
    _lib._lib = None
    try:
        with pytest.raises(RuntimeError):
            _lib.load(str(tmp_path / "nope.so"))
    finally:
        _lib._lib = saved


# ----------------------------------------------------------------- rejections (no GPU)

no_gpu = pytest.mark.skipif(torch.cuda.is_available(),
                            reason="fake device addresses are only used where no GPU exists")
FAKE = 1 << 40  # 16-byte aligned, never dereferenced


def desc(T, H, D, stride=None, dtype=_lib.GDN_BF16, ptr=FAKE, ndim=3):
    d = _lib.GdnTensor()
    d.ptr = ptr
    d.ndim = ndim
    d.dtype = dtype
    shape = (T, H, D) if ndim == 3 else (1, T, H, D)
    st = stride or (H * D, D, 1)
    if ndim == 4:
        st = (T * H * D,) + tuple(st)
    for i, (a, b) in enumerate(zip(shape, st)):
        d.shape[i] = a
        d.stride[i] = b
    return d


def prefill(lib, q, k, v, o, cu, N, chunk=64, flags=0):
    cu_arr = (ctypes.c_int32 * len(cu))(*cu)
    return lib.gdn_chunk_prefill(ctypes.byref(q), ctypes.byref(k), ctypes.byref(v),
                                 FAKE, FAKE, FAKE, ctypes.cast(cu_arr, ctypes.c_void_p),
                                 N, chunk, 1.0, flags, None, ctypes.byref(o), None, None,
                                 0, None, None)


@no_gpu
def test_head_first_rejected_without_T_less_than_H_heuristic(lib):
    T, Hk, Hv, D = 12, 16, 32, 128
    q = desc(T, Hk, D, stride=(D, T * D, 1))          # head-first memory
    k, v, o = desc(T, Hk, D), desc(T, Hv, D), desc(T, Hv, D)
    assert prefill(lib, q, k, v, o, [0, T], 1) == 3   # GDN_ERR_LAYOUT


@no_gpu
def test_batched_4d_with_b_gt_1_rejected(lib):
    q = desc(8, 2, 128, ndim=4)
    q.shape[0] = 2
    k, v, o = desc(8, 2, 128), desc(8, 2, 128), desc(8, 2, 128)
    assert prefill(lib, q, k, v, o, [0, 8], 1) == 3


@no_gpu
@pytest.mark.parametrize("cu", [[1, 8], [0, 9], [0, 5, 3, 8]])
def test_bad_cu_seqlens_rejected(lib, cu):
    q, k, v, o = desc(8, 2, 128), desc(8, 2, 128), desc(8, 2, 128), desc(8, 2, 128)
    assert prefill(lib, q, k, v, o, cu, len(cu) - 1) == 5


@no_gpu
def test_shape_and_dtype_mismatches_rejected(lib):
    q, k, o = desc(8, 2, 128), desc(8, 2, 128), desc(8, 3, 128)
    v = desc(8, 3, 128)
    assert prefill(lib, q, k, v, o, [0, 8], 1) == 2            # Hv % Hk != 0
    v = desc(8, 2, 128, dtype=_lib.GDN_F32)
    assert prefill(lib, q, k, v, desc(8, 2, 128), [0, 8], 1) == 4
    q2 = desc(8, 2, 128, ptr=FAKE + 2)                       # misaligned
    assert prefill(lib, q2, k, desc(8, 2, 128), desc(8, 2, 128), [0, 8], 1) == 3


@no_gpu
def test_unsupported_shapes_rejected(lib):
    q, k, v, o = desc(8, 2, 96), desc(8, 2, 96), desc(8, 2, 96), desc(8, 2, 96)
    assert prefill(lib, q, k, v, o, [0, 8], 1) == 6
    q, k, v, o = desc(8, 2, 64), desc(8, 2, 64), desc(8, 2, 64), desc(8, 2, 64)
    dq = ctypes.byref
    rc = lib.gdn_recurrent_decode(dq(q), dq(k), dq(v), FAKE, FAKE, FAKE, 8, None, 1.0, 0,
                                  dq(o), None, None)
    assert rc == 6


@no_gpu
def test_conv_rejections(lib):
    cu = (ctypes.c_int32 * 2)(0, 8)
    cup = ctypes.cast(cu, ctypes.c_void_p)
    assert lib.gdn_conv1d_fwd(FAKE, 8, 12, FAKE, None, FAKE, cup, 1, None, None, FAKE,
                              None) == 6                        # C % 8 != 0
    assert lib.gdn_conv1d_fwd(FAKE, 8, 16, None, None, FAKE, cup, 1, None, None, FAKE,
                              None) == 1                        # no weights
    assert lib.gdn_conv1d_update(FAKE, 4, 16, FAKE, None, FAKE, 2, None, FAKE, None,
                                 None) == 2                     # P < N without indices


@no_gpu
def test_fused_decode_rejections(lib):
    vp = None
    args = dict(x=FAKE, N=4, Hk=2, Hv=6, dk=128, dv=128, w=FAKE, bias=vp, cs=FAKE, a=FAKE,
                b=FAKE, state=FAKE, P=4, idx=vp, scale=1.0, flags=0, o=FAKE, status=vp,
                stream=vp)

    def call(**kw):
        a = dict(args, **kw)
        return lib.gdn_fused_decode(a["x"], a["N"], a["Hk"], a["Hv"], a["dk"], a["dv"],
                                    a["w"], a["bias"], a["cs"], a["a"], a["b"], a["state"],
                                    a["P"], a["idx"], a["scale"], a["flags"], a["o"],
                                    a["status"], a["stream"])

    assert call(Hv=5) == 2                 # Hv % Hk != 0
    assert call(dk=64, dv=64) == 6         # only d = 128
    assert call(a=None) == 1               # no gate logits
    assert call(P=3) == 2                  # P < N without indices
    assert call(o=FAKE + 8) == 3           # misaligned output
    assert call(N=0, x=None) == 0          # nothing to do


@no_gpu
def test_workspace_size(lib):
    """The CUDA-core path needs no workspace; the tensor-core path needs one tile per
    (chunk slot, v-head), the bf16 128x64 [Lo ; Mt] tile plus four fp32 per-token
    scalars, over ceil(T / 64) + N + 1 slots (chunks anchored at every sequence start)."""
    f = lib.gdn_chunk_prefill_workspace_size
    assert f(2, 500, 2, 4, 64, 64, 64, 0) == 0
    assert f(2, 500, 2, 4, 128, 128, 16, 0) == 0
    assert f(2, 500, 2, 4, 128, 128, 64, _lib.GDN_PREFILL_SIMT) == 0
    tile = 128 * 64 * 2 + 4 * 64 * 4
    for N, T, Hv in ((1, 4096, 48), (8, 30702, 48), (40, 311605, 32), (3, 0, 6)):
        assert f(N, T, 16, Hv, 128, 128, 64, 0) == (-(-T // 64) + N + 1) * Hv * tile


def cp_prefill(lib, q, k, v, o, cu, N, range_chunks, ws=None, ws_bytes=0):
    cu_arr = (ctypes.c_int32 * len(cu))(*cu)
    return lib.gdn_chunk_prefill_cp(ctypes.byref(q), ctypes.byref(k), ctypes.byref(v),
                                    FAKE, FAKE, FAKE, ctypes.cast(cu_arr, ctypes.c_void_p),
                                    N, 64, 1.0, 0, range_chunks, None, ctypes.byref(o), None,
                                    ws, ws_bytes, None, None)


@no_gpu
def test_cp_workspace_size(lib):
    """The context-parallel scan's scratch: the workspace tiles of the split batch (one
    range per range_chunks chunks of each sequence, at least one), then three
    [ranges, Hv, dk, dv] fp32 state arrays (end states from the first pass, transition
    maps, composed start states) and three int32 tables, each 256-byte aligned."""
    f = lib.gdn_chunk_prefill_cp_workspace_size
    lens = [700, 64, 1, 300, 129, 0]
    cu = [0]
    for n in lens:
        cu.append(cu[-1] + n)
    cu_arr = (ctypes.c_int32 * len(cu))(*cu)
    cup = ctypes.cast(cu_arr, ctypes.c_void_p)
    T, N, Hv = cu[-1], len(lens), 6

    def a256(x):
        return (x + 255) // 256 * 256
    for rc in (1, 2, 5, 100):
        nr = sum(max(1, -(-(-(-n // 64)) // rc)) for n in lens)
        tiles = (-(-T // 64) + nr + 1) * Hv * (128 * 64 * 2 + 4 * 64 * 4)
        want = (a256(tiles) + 3 * a256(nr * Hv * 128 * 128 * 4) + a256((nr + 1) * 4) +
                a256(nr * 4) + a256(N * 4))
        assert f(cup, N, T, 2, Hv, 128, 128, 64, rc) == want, rc
    assert f(cup, N, T, 2, Hv, 128, 128, 64, 0) == 0       # no range length
    assert f(cup, N, T, 2, Hv, 64, 64, 64, 2) == 0         # not a tensor-core shape


@no_gpu
def test_cp_rejections(lib):
    q, k, v, o = desc(8, 2, 128), desc(8, 2, 128), desc(8, 2, 128), desc(8, 2, 128)
    assert cp_prefill(lib, q, k, v, o, [0, 8], 1, 0) == 2     # range_chunks < 1
    assert cp_prefill(lib, q, k, v, o, [0, 8], 1, 2) == 9     # no workspace
    f32 = [desc(8, 2, 128, dtype=_lib.GDN_F32) for _ in range(4)]
    assert cp_prefill(lib, *f32, [0, 8], 1, 2) == 6           # CUDA-core shapes only
    qh = desc(8, 2, 128, stride=(128, 8 * 128, 1))            # head-first
    assert cp_prefill(lib, qh, k, v, o, [0, 8], 1, 2) == 3


def test_cp_range_hint_model(lib):
    """The range hint's wave-count model with an explicit SM count (no device needed).  On
    152 SMs it picks, for each single-sequence shape below, the range length measured
    fastest on the GB300 among the plain scan and the timed splits (times in us, mean of
    20 runs with L2 flushed between them):
    32768 tokens x 6 v-heads: 40 chunks (303; plain 854, 43 -> 317, 74 -> 343);
    65536 x 3: 40 (324; plain 1636, 43 -> 336, 74 -> 355); 65536 x 1: 27 (193; 32 -> 201);
    32768 x 12: 74 (530; 47 -> 571); 32768 x 4: 26 (225; 47 -> 237);
    16384 x 24: 86 (434; 64 -> 474, plain 510); 16384 x 12: 37 (286; 64 -> 306);
    16384 x 8: 26 (209; 43 -> 217); 16384 x 1: 13 (96; 16 -> 100);
    8192 x 6: 19 (114; 11 -> 115); 4096 x 24: 22 (135; plain 140, 13 -> 188).
    The 27B layer's 4096 tokens over 48 v-heads and any single-chunk sequence stay plain
    (4096 x 48: plain 165, 64 -> 186).  Every SM count gets a valid range length (or 0),
    and bad arguments answer 0."""
    f = lib.gdn_chunk_prefill_cp_range_hint_for
    measured_best = {(32768, 6): 40, (65536, 3): 40, (65536, 1): 27, (32768, 12): 74,
                     (32768, 4): 26, (16384, 24): 86, (16384, 12): 37, (16384, 8): 26,
                     (16384, 1): 13, (8192, 6): 19, (4096, 24): 22, (4096, 48): 0}
    for (L, Hv), r in measured_best.items():
        assert f(L, Hv, 152) == r, (L, Hv, f(L, Hv, 152), r)
    assert f(64, 6, 152) == 0 and f(1, 1, 152) == 0
    assert f(32768, 6, 0) == 0 and f(0, 6, 152) == 0 and f(32768, 0, 152) == 0
    for sms in (8, 32, 76, 152, 304):
        r = f(32768, 6, sms)
        assert 0 <= r < 512
    # a sequence whose chains fill the device on their own is never split
    assert f(4096, 64, 64) == 0


def test_cp_range_hint_without_device(lib):
    """The range hint is a host-side estimate that needs the device's SM count: without a
    current device, and for arguments that are not positive, it answers 0 (the plain
    scan)."""
    import torch
    f = lib.gdn_chunk_prefill_cp_range_hint
    assert f(0, 6) == 0 and f(-5, 6) == 0 and f(4096, 0) == 0
    if not torch.cuda.is_available():
        assert f(32768, 6) == 0


def test_selftest_needs_a_status_word(lib):
    assert lib.gdn_selftest_bounded_wait(None, None) == 1   # GDN_ERR_NULL, nothing launched


def test_layer_prefill_rejections(lib):
    cu = (ctypes.c_int32 * 2)(0, 8)
    cup = ctypes.cast(cu, ctypes.c_void_p)
    bad = (ctypes.c_int32 * 2)(0, 9)
    badp = ctypes.cast(bad, ctypes.c_void_p)

    def call(x=FAKE, T=8, Hk=2, Hv=6, cu_h=cup, y=FAKE, w=FAKE):
        return lib.gdn_layer_prefill(x, T, Hk, Hv, 128, 128, w, None, FAKE, cu_h, 1, None,
                                     None, y, FAKE, FAKE, 1.0, 0, None, FAKE, None, None, 0,
                                     None, None, None)

    assert call(Hk=0) == 2                 # no heads
    assert call(w=None) == 1               # no conv weights
    assert call(y=None) == 1               # nowhere to put the conv output
    assert call(cu_h=badp) == 5            # cu_seqlens[N] != T
    assert call(x=FAKE + 4) == 3           # misaligned input


def test_forced_error_env(monkeypatch):
    """GDN_FORCE_ERROR makes the named binding entries raise the given status at once,
    before any argument or device check (host-side fault injection)."""
    import torch
    gdn = pytest.importorskip("gated_deltanet_linear_11_gb300")
    z = torch.zeros(1)
    monkeypatch.setenv("GDN_FORCE_ERROR", "gdn_chunk_prefill=7, gdn_fused_decode=10")
    with pytest.raises(gdn.GdnError) as e:
        gdn.gdn_chunk_prefill(z, z, z, z, z, z)
    assert e.value.code == 7 and "GDN_FORCE_ERROR" in str(e.value)
    with pytest.raises(gdn.GdnError) as e:
        gdn.gdn_fused_decode(z, z, None, z, z, z, z, 1, 1, 128, 128)
    assert e.value.code == 10
    # entries not named run their own checks (here: CPU tensors are refused)
    with pytest.raises(ValueError):
        gdn.gdn_recurrent_decode(z, z, z, z, z, z)
    monkeypatch.setenv("GDN_FORCE_ERROR", "gdn_chunk_prefill")
    with pytest.raises(ValueError):
        gdn.gdn_chunk_prefill(z, z, z, z, z, z)
    monkeypatch.delenv("GDN_FORCE_ERROR")
    with pytest.raises(ValueError):
        gdn.gdn_chunk_prefill(z, z, z, z, z, z)


def test_debug_env_sets_the_finite_check_flag(monkeypatch):
    """GDN_DEBUG turns on GDN_CHECK_INPUTS for every call that takes flags; the flag is a
    bit of its own, and its status has a name."""
    gdn = pytest.importorskip("gated_deltanet_linear_11_gb300")
    monkeypatch.delenv("GDN_DEBUG", raising=False)
    assert gdn._debug_flags() == 0
    monkeypatch.setenv("GDN_DEBUG", "0")
    assert gdn._debug_flags() == 0
    monkeypatch.setenv("GDN_DEBUG", "1")
    assert gdn._debug_flags() == _lib.GDN_CHECK_INPUTS == 0x1000
    others = (_lib.GDN_QK_L2NORM, _lib.GDN_PREFILL_SIMT, _lib.GDN_PREFILL_TILES2,
              _lib.GDN_PREFILL_TILES3, _lib.GDN_LAYER_FUSED_VCONV)
    assert all(f & _lib.GDN_CHECK_INPUTS == 0 for f in others)
    assert _lib.STATUS[11] == "GDN_ERR_NONFINITE"
    text = open(os.path.join(ROOT, "include", "gdn.h")).read()
    assert "#define GDN_CHECK_INPUTS 0x1000u" in text and "GDN_ERR_NONFINITE = 11" in text
