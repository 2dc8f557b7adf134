"""Host-side checks of the C ABI: the library loads, exports every declared
symbol, and the host-only entry points (page pool, checkpoint count, byte
ratio, argument validation) behave as documented.  Nothing here launches a
kernel: every validation case fails before any launch, and fake device
pointers are never dereferenced.
"""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "kda.h")


@pytest.fixture(scope="module")
def K():
    from kda_delta_rule_gb300 import build
    build.build()
    from kda_delta_rule_gb300 import kda
    return kda


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(kda_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for must in ("kda_decode_step", "kda_verify_replay", "kda_prefill_chunked",
                 "kda_pack_heads", "kda_unpack_heads", "kda_num_checkpoints",
                 "kda_pool_create", "kda_pool_alloc", "kda_pool_free",
                 "kda_store_kda", "kda_load_kda", "kda_snapshot_cost_ratio"):
        assert must in names


def test_library_exports_every_declared_symbol(K):
    lib = ctypes.CDLL(K._LIB_PATH)
    missing = [n for n in declared_functions() if not hasattr(lib, n)]
    assert not missing, missing


def test_status_strings(K):
    assert K._lib.kda_status_string(0) == b"KDA_OK"
    assert K._lib.kda_status_string(-7) == b"KDA_ERR_ALIAS"
    assert K._lib.kda_version() >= 1


def test_chain_columns_knob(K):
    f = K._lib.kda_set_prefill_chain_columns
    for bad in (-1, 1, 16, 48, 128):
        assert f(bad) == -1
    for good in (32, 64, 0):
        assert f(good) == 0
    with pytest.raises(K.KdaError):
        K.kda_set_prefill_chain_columns(96)
    K.kda_set_prefill_chain_columns(0)


def test_snapshot_cost_ratio_matches_pages(K):
    assert round(K.kda_snapshot_cost_ratio(2, 8, 8), 2) == 1.94
    assert round(K.kda_snapshot_cost_ratio(1, 16, 16), 2) == 3.94
    assert K.kda_snapshot_cost_ratio(16, 32, 32) == pytest.approx(1024 / 129)
    with pytest.raises(ValueError):
        K.kda_snapshot_cost_ratio(0, 8, 8)


def test_num_checkpoints(K):
    assert K.kda_num_checkpoints(None, 8192, 512) == 16
    assert K.kda_num_checkpoints([0, 8192, 9192, 9703], 9703, 512) == 16 + 1 + 0
    assert K.kda_num_checkpoints([0, 100], 100, 0) == 0
    with pytest.raises(K.KdaError):
        K.kda_num_checkpoints([0, 50, 40], 40, 64)     # decreasing
    with pytest.raises(K.KdaError):
        K.kda_num_checkpoints([0, 50], 60, 64)         # does not end at T


def _fake_pool(K, page_bytes=4096, n_pages=8):
    h = ctypes.c_void_p()
    base = ctypes.c_void_p(0x10000)          # never dereferenced by the pool
    assert K._lib.kda_pool_create(base, page_bytes, n_pages, ctypes.byref(h)) == 0
    return h


def test_pool_single_free_list_two_kinds(K):
    lib = K._lib
    h = _fake_pool(K)
    ids = (ctypes.c_int32 * 8)()
    assert lib.kda_pool_alloc(h, K.PAGE_KDA_STATE, 3, ids) == 0
    assert list(ids[:3]) == [0, 1, 2]
    assert lib.kda_pool_alloc(h, K.PAGE_MLA_KV, 2, ctypes.byref(ids, 12)) == 0
    assert list(ids[3:5]) == [3, 4]
    assert lib.kda_pool_num_free(h) == 3
    assert lib.kda_pool_page_kind(h, 1) == K.PAGE_KDA_STATE
    assert lib.kda_pool_page_kind(h, 4) == K.PAGE_MLA_KV
    assert lib.kda_pool_page_ptr(h, 2) == 0x10000 + 2 * 4096
    # all-or-nothing when the pool is short
    more = (ctypes.c_int32 * 4)()
    assert lib.kda_pool_alloc(h, K.PAGE_KDA_STATE, 4, more) == -6
    assert lib.kda_pool_num_free(h) == 3
    # free returns pages to the one list; lowest index first again
    back = (ctypes.c_int32 * 2)(1, 3)
    assert lib.kda_pool_free(h, 2, back) == 0
    assert lib.kda_pool_page_kind(h, 1) == K.PAGE_FREE
    one = (ctypes.c_int32 * 1)()
    assert lib.kda_pool_alloc(h, K.PAGE_MLA_KV, 1, one) == 0 and one[0] == 1
    # freeing a free page (or a page twice) is rejected and frees nothing
    bad = (ctypes.c_int32 * 2)(0, 3)
    assert lib.kda_pool_free(h, 2, bad) == -1
    assert lib.kda_pool_page_kind(h, 0) == K.PAGE_KDA_STATE
    dup = (ctypes.c_int32 * 2)(0, 0)
    assert lib.kda_pool_free(h, 2, dup) == -1
    assert lib.kda_pool_destroy(h) == 0


def test_store_kda_requires_a_state_page(K):
    lib = K._lib
    h = _fake_pool(K, page_bytes=4096, n_pages=2)
    ids = (ctypes.c_int32 * 1)()
    assert lib.kda_pool_alloc(h, K.PAGE_MLA_KV, 1, ids) == 0
    S = ctypes.c_void_p(0x20000)
    assert lib.kda_store_kda(h, ids[0], S, 1024, 1024, 1, 1, 32, 32, None) == -1   # wrong kind
    assert lib.kda_store_kda(h, 1, S, 1024, 1024, 1, 1, 32, 32, None) == -1        # free page
    assert lib.kda_pool_alloc(h, K.PAGE_KDA_STATE, 1, ids) == 0
    assert lib.kda_store_kda(h, ids[0], S, 4096, 4096, 1, 1, 64, 64, None) == -2   # too big
    lib.kda_pool_destroy(h)


# ---------------------------------------------------------------------------
# Validation (every case fails before a launch)
# ---------------------------------------------------------------------------
A = 0x100000          # fake 16-byte aligned device addresses, never dereferenced


def P(off):
    return ctypes.c_void_p(A + off)


def test_decode_validation(K):
    f = K._lib.kda_decode_step
    base = [P(0), P(1 << 20), P(2 << 20), P(3 << 20), P(4 << 20), P(5 << 20), P(6 << 20)]
    assert f(*base, 2, 2, 48, 32, 0, 0, None) == -2          # unsupported dk
    assert f(*base, 2, 2, 32, 32, 7, 0, None) == -3          # dtype
    assert f(*base, 2, 2, 32, 32, 0, 5, None) == -1          # mode
    assert f(None, *base[1:], 2, 2, 32, 32, 0, 0, None) == -1
    bad = list(base); bad[0] = P(4)
    assert f(*bad, 2, 2, 32, 32, 0, 0, None) == -4           # misaligned state
    alias = list(base); alias[6] = P(64)
    assert f(*alias, 2, 2, 32, 32, 0, 0, None) == -7         # o inside S
    assert f(*base, 0, 2, 32, 32, 0, 0, None) == 0           # empty batch: no-op
    assert b"32, 64 or 128" in K._lib.kda_last_error() or True


def test_replay_rejects_writing_the_committed_state(K):
    f = K._lib.kda_verify_replay
    S_c, S_new = P(0), P(0)
    args = [S_c, P(1 << 20), P(2 << 20), P(3 << 20), P(4 << 20), P(5 << 20), P(6 << 20), S_new,
            P(7 << 20)]
    assert f(*args, 4, 2, 2, 32, 32, 0, 0, None) == -7
    args[7] = P(1024)                                         # partial overlap
    assert f(*args, 4, 2, 2, 32, 32, 0, 0, None) == -7
    args[7] = P(8 << 20)
    assert f(*args, 0, 2, 2, 32, 32, 0, 0, None) == -2        # draft 0
    assert f(*args, 17, 2, 2, 32, 32, 0, 0, None) == -2       # draft > 16


def test_replay_layers_validation(K):
    f = K._lib.kda_verify_replay_layers
    # layers x B x H x 32 x 32 fp32 = 3 x 4096 B per (b, h): S_new inside the stacked S_committed
    args = [P(0), P(1 << 20), P(2 << 20), P(3 << 20), P(4 << 20), P(5 << 20), P(6 << 20), P(4096 * 2),
            P(7 << 20)]
    assert f(3, *args, 4, 1, 1, 32, 32, 0, 0, None) == -7
    args[7] = P(8 << 20)
    assert f(-1, *args, 4, 1, 1, 32, 32, 0, 0, None) == -2
    assert f(0, *args, 4, 1, 1, 32, 32, 0, 0, None) == 0      # no layers: no-op
    assert f(2, *args, 0, 1, 1, 32, 32, 0, 0, None) == -2     # draft 0


def test_slot_entries_validation(K):
    """kda_decode_step_slots / kda_verify_replay_slots reject bad layouts, empty pools,
    missing slot ids and pool aliasing before any launch."""
    d = K._lib.kda_decode_step_slots
    proj = [P(1 << 24), P(2 << 24), P(3 << 24), P(4 << 24), P(5 << 24), P(6 << 24)]
    # (S_pool, n_slots, slot_ids, layout, q, k, v, g, beta, o, B, H, dk, dv, dtype, mode, stream)
    assert d(P(0), 8, P(7 << 24), 2, *proj, 4, 2, 32, 32, 0, 0, None) == -1      # layout
    assert d(P(0), 0, P(7 << 24), 0, *proj, 4, 2, 32, 32, 0, 0, None) == -2      # no slots
    assert d(P(0), 8, None, 1, *proj, 4, 2, 32, 32, 0, 0, None) == -1            # slot ids NULL
    assert d(P(8), 8, P(7 << 24), 1, *proj, 4, 2, 32, 32, 0, 0, None) == -4      # unaligned pool
    o_in_pool = proj[:5] + [P(4096)]
    assert d(P(0), 8, P(7 << 24), 1, *o_in_pool, 4, 2, 32, 32, 0, 0, None) == -7
    assert d(P(0), 8, P(7 << 24), 1, *proj, 0, 2, 32, 32, 0, 0, None) == 0       # B = 0: no-op
    r = K._lib.kda_verify_replay_slots
    pr = [P(1 << 24), P(2 << 24), P(3 << 24), P(4 << 24), P(5 << 24)]

    def rep(pool, pool_new, s_in, s_out, layout=1, n_slots=8, layers=2, draft=4):
        # (layers, S_pool, S_pool_new, n_slots, slot_in, slot_out, layout, q, k, v, g, beta,
        #  n_accepted, out, draft, B, H, dk, dv, dtype, mode, stream)
        return r(layers, pool, pool_new, n_slots, s_in, s_out, layout, *pr, P(6 << 24), P(9 << 24),
                 draft, 4, 2, 32, 32, 0, 0, None)

    assert rep(P(0), P(0), P(7 << 24), None) == -7            # same pool, same slots
    assert rep(P(0), P(0), P(7 << 24), P(7 << 24)) == -7      # same pool, same id array
    assert rep(P(0), P(4096), P(7 << 24), P(8 << 24)) == -7   # pools partly overlap
    assert rep(P(0), P(8 << 20), P(7 << 24), None, layout=3) == -1
    assert rep(P(0), P(8 << 20), None, None) == -1
    assert rep(P(0), P(8 << 20), P(7 << 24), None, draft=17) == -2
    assert rep(P(0), P(8 << 20), P(7 << 24), None, layers=0) == 0


def test_prologue_entries_validation(K):
    """kda_input_prep / kda_decode_step_fused: kernel size, activation, g_min, partial
    projection outputs and aliasing are rejected before any launch."""
    f = K._lib.kda_input_prep
    cu = (ctypes.c_int32 * 3)(0, 40, 100)

    def prep(**kw):
        a = dict(mixed=P(1 << 24), wt=P(2 << 24), w=4, win_in=None, win_out=None, gl=P(3 << 24), bl=P(4 << 24),
                 g_min=-5.0, act=1, cu=cu, n=2, T=100, H=2, dk=32, dv=32, dtype=0, q=P(5 << 24), k=P(6 << 24),
                 v=P(7 << 24), g=P(8 << 24), beta=P(9 << 24), stride=0, ck=None, nck=0)
        a.update(kw)
        return f(a["mixed"], a["wt"], a["w"], a["win_in"], a["win_out"], a["gl"], a["bl"], a["g_min"], a["act"],
                 a["cu"], a["n"], a["T"], a["H"], a["dk"], a["dv"], a["dtype"], a["q"], a["k"], a["v"], a["g"],
                 a["beta"], a["stride"], a["ck"], a["nck"], None)

    assert prep(w=1) == -2 and prep(w=9) == -2
    assert prep(act=2) == -1
    assert prep(g_min=0.0) == -1
    assert prep(q=None) == -1
    assert prep(q=P((1 << 24) + 64)) == -7                      # q inside mixed
    assert prep(k=P((5 << 24) + 16)) == -7                      # k overlaps q
    assert prep(ck=P(10 << 24), stride=0) == -1
    assert prep(ck=P(10 << 24), stride=32, nck=1) == -2         # 1 + 1 checkpoints needed
    assert prep(T=101) == -2                                   # cu_seqlens does not end at T
    assert prep(H=0) == 0
    d = K._lib.kda_decode_step_fused

    def dec(**kw):
        a = dict(S=P(0), n_slots=0, slots=None, layout=0, conv=P(1 << 24), mixed=P(2 << 24), wt=P(3 << 24), w=4,
                 gl=P(4 << 24), bl=P(5 << 24), g_min=-5.0, act=1, o=P(6 << 24), qo=None, ko=None, vo=None,
                 go=None, bo=None, B=2, H=2, dk=32, dv=32, dtype=0, mode=0)
        a.update(kw)
        return d(a["S"], a["n_slots"], a["slots"], a["layout"], a["conv"], a["mixed"], a["wt"], a["w"], a["gl"],
                 a["bl"], a["g_min"], a["act"], a["o"], a["qo"], a["ko"], a["vo"], a["go"], a["bo"], a["B"], a["H"],
                 a["dk"], a["dv"], a["dtype"], a["mode"], None)

    assert dec(qo=P(7 << 24)) == -1                            # only some projection outputs
    assert dec(layout=5) == -1
    assert dec(slots=P(8 << 24), n_slots=0) == -2
    assert dec(conv=P(64)) == -7                                # conv window inside S
    assert dec(w=5) == -2                                       # fused decode keeps w <= 4
    assert dec(conv=None) == -1
    assert dec(B=0) == 0


def test_prefill_validation(K):
    f = K._lib.kda_prefill_chunked
    cu = (ctypes.c_int32 * 3)(0, 100, 228)

    def call(**kw):
        a = dict(S0=P(0), q=P(1 << 24), k=P(2 << 24), v=P(3 << 24), g=P(4 << 24), beta=P(5 << 24),
                 cu=cu, n=2, T=228, H=2, dk=32, dv=32, dtype=0, chunk=64, stride=64,
                 o=P(6 << 24), Sf=P(7 << 24), pool=P(8 << 24), page_bytes=8192,
                 ids=P(9 << 24), pos=None, nck=10, ws=None, ws_bytes=0, mode=0)
        a.update(kw)
        return f(a["S0"], a["q"], a["k"], a["v"], a["g"], a["beta"], a["cu"], a["n"], a["T"],
                 a["H"], a["dk"], a["dv"], a["dtype"], a["chunk"], a["stride"], a["o"], a["Sf"],
                 a["pool"], a["page_bytes"], a["ids"], a["pos"], a["nck"], a["ws"], a["ws_bytes"],
                 a["mode"], None)

    assert call(chunk=32) == -1
    assert call(stride=96) == -1                               # not a multiple of chunk
    assert call(T=229) == -2                                   # cu_seqlens does not end at T
    assert call(cu=(ctypes.c_int32 * 3)(0, 120, 100), T=100) == -2
    assert call(nck=1) == -2                                   # 1 + 2 checkpoints needed
    assert call(page_bytes=4096) == -2                         # page smaller than H*dk*dv*4
    assert call(ids=None) == -1
    assert call(Sf=P(64)) == -7                                # S_final overlaps S0
    assert call(o=P(1 << 24)) == -7                            # o overlaps q
    assert call(cu=None, n=2) == -1
    assert call(H=0) == 0                                      # nothing to do
    # tensor-core shapes need the workspace that kda_prefill_workspace_bytes reports
    need = K._lib.kda_prefill_workspace_bytes(cu, 2, 228, 2, 128, 128, 1)
    assert need == (2 + 2) * 2 * 74240                         # ceil(100/64)+ceil(128/64) chunks x H
    assert K._lib.kda_prefill_workspace_bytes(cu, 2, 228, 2, 32, 32, 1) == 0
    assert K._lib.kda_prefill_workspace_bytes(cu, 2, 228, 2, 128, 128, 0) == 0
    assert call(dk=128, dv=128, dtype=1, page_bytes=2 * 128 * 128 * 4, ws=P(10 << 24),
                ws_bytes=need - 16) == -2
    assert call(dk=128, dv=128, dtype=1, page_bytes=2 * 128 * 128 * 4, ws=P(10 << 24) if False else
                ctypes.c_void_p(A + (10 << 24) + 8), ws_bytes=need) == -4


def test_prefill_host_validation(K):
    lib = K._lib
    assert lib.kda_prefill_host_scratch_bytes(2, 32, 32, 0, 0, 100) > 0
    assert lib.kda_prefill_host_scratch_bytes(2, 32, 32, 0, 96, 100) == -1   # stride not a multiple of 64
    assert lib.kda_prefill_host_scratch_bytes(2, 48, 32, 0, 0, 100) == -2
    need = lib.kda_prefill_host_scratch_bytes(2, 32, 32, 0, 0, 256)
    cu = (ctypes.c_int32 * 3)(0, 100, 228)
    f = lib.kda_prefill_chunked_host

    def call(scratch, nbytes, chunk=64):
        # host buffers are never touched: validation fails first
        return f(None, P(1 << 20), P(2 << 20), P(3 << 20), P(4 << 20), P(5 << 20), cu, 2, 228, 2, 32, 32, 0,
                 chunk, 0, P(6 << 20), P(7 << 20), None, 0, None, None, 0, scratch, nbytes, 256, 0, None)
    assert call(P(8 << 20), need - 256) == -2                # scratch too small
    assert call(ctypes.c_void_p(A + (8 << 20) + 16), need) == -4   # not 256-byte aligned
    assert call(P(8 << 20), need, chunk=32) == -1


def test_ring_host_side(K):
    lib = K._lib
    assert lib.kda_ring_bytes(4, 2, 3, 32, 32, 0) > 0
    assert lib.kda_ring_bytes(0, 2, 3, 32, 32, 0) == -2
    assert lib.kda_ring_bytes(17, 2, 3, 32, 32, 0) == -2       # capacity above KDA_MAX_DRAFT
    h = ctypes.c_void_p()
    assert lib.kda_ring_create(P(16), 4, 2, 3, 32, 32, 0, ctypes.byref(h)) == -4   # not 256-aligned
    assert lib.kda_ring_create(P(0), 4, 2, 3, 32, 32, 0, ctypes.byref(h)) == 0     # never dereferenced here
    assert lib.kda_ring_len(h) == 0
    assert lib.kda_verify_replay_ring(h, P(1 << 20), P(2 << 20), P(3 << 20), P(4 << 20), 0, None) == -2  # empty
    assert lib.kda_ring_reset(h) == 0
    assert lib.kda_ring_destroy(h) == 0


def test_pack_validation(K):
    f = K._lib.kda_pack_heads
    assert f(P(0), 4096, 1024, P(1 << 20), 100, 2, 2, 32, 32, None) == -2   # flat too small
    assert f(P(0), 4098, 1024, P(1 << 20), 8192, 2, 2, 32, 32, None) == -4  # stride % 4
    assert f(P(8), 4096, 1024, P(1 << 20), 8192, 2, 2, 32, 32, None) == -4  # misaligned


def test_prefill_scan_validation(K):
    # every call below carries one defect, so it is refused before any launch
    lib = K._lib
    T, H, d = 4096, 2, 128
    need = lib.kda_prefill_scan_workspace_bytes(T, H, d, d, 1, 512, 4)
    cu = (ctypes.c_int32 * 2)(0, T)
    assert need > lib.kda_prefill_workspace_bytes(cu, 1, T, H, d, d, 1) > 0   # images, then the piece states
    assert lib.kda_prefill_scan_workspace_bytes(T, H, d, d, 1, 96, 4) == -1     # stride not a multiple of 64
    assert lib.kda_prefill_scan_workspace_bytes(T, H, d, d, 1, 512, 257) == -1  # more than 256 pieces
    assert lib.kda_prefill_scan_workspace_bytes(T, H, d, d, 1, 512, -1) == -1
    assert lib.kda_prefill_scan_workspace_bytes(T, H, 32, 32, 1, 512, 4) == -2  # no tensor-core kernels there
    assert lib.kda_prefill_scan_workspace_bytes(T, H, d, d, 0, 512, 4) == -2    # fp32: the CUDA-core path only
    f = lib.kda_prefill_scan

    def call(**kw):
        a = dict(S0=P(0), q=P(1 << 24), k=P(2 << 24), v=P(3 << 24), g=P(4 << 24), beta=P(5 << 24), T=T, H=H,
                 dk=d, dv=d, dtype=1, chunk=64, stride=512, o=P(6 << 24), Sf=P(7 << 24), pool=P(8 << 24),
                 page_bytes=H * d * d * 4, ids=P(9 << 24), pos=None, nck=8, ws=P(10 << 24), ws_bytes=need,
                 segments=4, mode=0)
        a.update(kw)
        return f(a["S0"], a["q"], a["k"], a["v"], a["g"], a["beta"], a["T"], a["H"], a["dk"], a["dv"],
                 a["dtype"], a["chunk"], a["stride"], a["o"], a["Sf"], a["pool"], a["page_bytes"], a["ids"],
                 a["pos"], a["nck"], a["ws"], a["ws_bytes"], a["segments"], a["mode"], None)

    assert call(ws_bytes=need - 256) == -2                     # workspace too small
    assert call(ws=None) == -2
    assert call(ws=ctypes.c_void_p(A + (10 << 24) + 16)) == -4  # not 256-byte aligned
    assert call(chunk=32) == -1
    assert call(nck=7) == -2                                   # 8 checkpoints at 512 .. 4096
    assert call(ids=None) == -1
    assert call(Sf=P(64)) == -7                                # S_final overlaps S0
    assert call(segments=300) == -1


def test_noalloc_refuses_calls_past_its_scratch_before_any_device_call(K):
    lib = K._lib
    T, H, d = 2048, 32, 128                                    # 32 chunks x 32 heads of chunk images
    cu = (ctypes.c_int32 * 2)(0, T)
    assert lib.kda_prefill_workspace_bytes(cu, 1, T, H, d, d, 1) > (64 << 20)
    st = lib.kda_prefill_chunked_noalloc(P(0), P(1 << 26), P(2 << 26), P(3 << 26), P(4 << 26), P(5 << 26), cu, 1,
                                         T, H, d, d, 1, 64, 512, P(6 << 26), P(7 << 26), P(8 << 26),
                                         H * d * d * 4, P(9 << 26), None, 4, 0, None)
    assert st == -2
    assert b"scratch" in lib.kda_last_error()
