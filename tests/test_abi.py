"""The C-ABI library loads and exports every symbol include/mla.h declares, and
host-side validation rejects bad arguments before anything is launched. CPU only:
no call here reaches a kernel launch."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "mla.h")


def _declared():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(mla_[a-z0-9_]+)\s*\(", src)))


@pytest.fixture(scope="module")
def lib():
    from mla_latent_kv_13_gb300 import build
    build.build()
    return ctypes.CDLL(build.LIB)


def test_header_declares_the_boundary():
    names = _declared()
    for n in ["mla_append_kv", "mla_decode_attention", "mla_decode_combine", "mla_absorb_q",
              "mla_out_absorb", "mla_decode_workspace_size", "mla_check_device_status",
              "mla_status_string"]:
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    for n in _declared():
        assert hasattr(lib, n), n


def test_binding_declares_every_symbol(lib):
    from mla_latent_kv_13_gb300 import mla
    assert sorted(mla.EXPORTED) == _declared()


def test_status_strings(lib):
    lib.mla_status_string.restype = ctypes.c_char_p
    assert lib.mla_status_string(0) == b"MLA_OK"
    assert lib.mla_status_string(4) == b"MLA_ERR_OUT_OF_RANGE"


def test_host_validation_rejects_before_launch(lib):
    vp = ctypes.c_void_p
    lib.mla_decode_attention.restype = ctypes.c_int
    null = vp(0)
    # null pointers
    rc = lib.mla_decode_attention(null, null, null, 1, null, 1, null, 1, 128, 64,
                                  ctypes.c_float(0.07), 0, null, ctypes.c_size_t(0), null, null,
                                  null)
    assert rc == 1
    # workspace sizes and unsupported head counts (pure host arithmetic)
    sz = ctypes.c_size_t(0)
    assert lib.mla_decode_workspace_size(16, 128, 4096, 0, ctypes.byref(sz)) == 0
    assert sz.value >= 256
    assert lib.mla_decode_workspace_size(16, 48, 4096, 0, ctypes.byref(sz)) == 2
    assert lib.mla_decode_workspace_size(16, 128, 4096, 4, ctypes.byref(sz)) == 0
    assert sz.value >= 256 + 16 * 4 * 128 * 512 * 4
    assert lib.mla_append_kv_workspace_size(128, 7168, ctypes.byref(sz)) == 0
    assert lib.mla_append_kv_workspace_size(128, 7000, ctypes.byref(sz)) == 1
    assert lib.mla_absorb_q_workspace_size(128, 7168, 1536, 128, ctypes.byref(sz)) == 0
    assert lib.mla_out_absorb_workspace_size(128, 128, 7168, ctypes.byref(sz)) == 0


def test_decode_plan_reports_splits_and_launches(lib):
    from mla_latent_kv_13_gb300 import mla
    assert mla.decode_plan(16, 128, 4096, 1) == (1, 1)        # no merge
    assert mla.decode_plan(16, 128, 4096, 4) == (4, 2)        # decode + merge
    # far more tiles than one pass of resident clusters: the balanced schedule
    assert mla.decode_plan(4096, 128, 32768, 0) == (0, 3)
    s, n = mla.decode_plan(2, 128, 64, 0)                     # one tile per sequence
    assert s >= 1 and n == (1 if s == 1 else 2)
    i = ctypes.c_int(0)
    assert lib.mla_decode_plan(0, 128, 64, 0, ctypes.byref(i), None) == 1
    assert lib.mla_decode_plan(4, 48, 64, 0, None, None) == 2


def test_projection_launches_validation_and_partial_plan(lib):
    """Launch counts of the projection calls: argument rules, and with no visible device the
    plan that writes split-K partials for a finalize launch (append 2, absorb_q 4 or 6 with W_QR
    and RoPE separate above 128 sequences, out_absorb 3, the combined call both calls' sum)."""
    import torch
    from mla_latent_kv_13_gb300 import mla
    assert lib.mla_projection_launches(0, 7168, 1536, 128, None, None, None, None) == 1
    assert lib.mla_projection_launches(128, 7000, 1536, 128, None, None, None, None) == 1
    assert lib.mla_projection_launches(128, 7168, 1500, 128, None, None, None, None) == 1
    assert lib.mla_projection_launches(128, 7168, 1536, 48, None, None, None, None) == 2
    a, q, o, aq = mla.projection_launches(128, 7168, 1536, 128)
    assert a in (1, 2) and q in (3, 4) and o in (2, 3) and aq in (3, 4, 5, 6)
    assert mla.projection_launches(200, 7168, 1536, 128)[1] in (5, 6)
    if not torch.cuda.is_available():
        # no device: partials everywhere, the combined call runs the two calls
        assert mla.projection_launches(128, 7168, 1536, 128) == (2, 4, 3, 6)
        assert mla.projection_launches(200, 7168, 1536, 128) == (2, 6, 3, 8)


def test_decode_output_alignment_checked_before_launch(lib):
    """The attention output rows are written with 32-byte stores: an output pointer that is
    16- but not 32-byte aligned is rejected on the host (nothing below is dereferenced or
    launched: every call returns at its argument checks)."""
    f = lib.mla_decode_attention
    f.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int,
                  ctypes.c_void_p, ctypes.c_int, ctypes.c_void_p, ctypes.c_int, ctypes.c_int,
                  ctypes.c_int, ctypes.c_float, ctypes.c_int, ctypes.c_void_p, ctypes.c_size_t,
                  ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p]
    f.restype = ctypes.c_int
    base = 1 << 20  # a 256-byte-aligned stand-in address
    # two fixed splits need partial buffers that a 256-byte workspace cannot hold: a call that
    # got past the alignment check would stop at the workspace check, still before any launch
    args = lambda out: (base, base, base, 8, base, 2, base, 4, 128, 64, 0.07, 2, base,
                        256, out, base, None)
    assert f(*args(base)) == 3
    assert f(*args(base + 16)) == 1
    assert f(*args(base + 8)) == 1
    g = lib.mla_decode_attention_partial
    g.argtypes = f.argtypes
    g.restype = ctypes.c_int
    assert g(*args(base + 16)) == 1


def test_prepare_validation_before_launch(lib):
    """mla_decode_prepare checks its arguments and the workspace size on the host; a fixed
    split needs no schedule, so the call returns at once. (Every call below returns before
    anything is launched: the pointers are never dereferenced.)"""
    from mla_latent_kv_13_gb300 import mla
    f = lib.mla_decode_prepare
    f.argtypes = [ctypes.c_void_p, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                  ctypes.c_void_p, ctypes.c_size_t, ctypes.c_void_p]
    f.restype = ctypes.c_int
    ws, sl, big = 256, 512, 1 << 40
    assert f(None, 4, 128, 64, 0, ws, big, None) == 1
    assert f(sl, 0, 128, 64, 0, ws, big, None) == 1
    assert f(sl, 4, 48, 64, 0, ws, big, None) == 2
    assert f(sl, 4, 128, 64, 300, ws, big, None) == 1
    assert f(sl, 4, 128, 64, 0, 255, big, None) == 1
    need = mla.decode_workspace_size(4096, 128, 32768, 0)
    assert f(sl, 4096, 128, 32768, 0, ws, need - 1, None) == 3
    # a fixed split: nothing to prepare, nothing launched
    assert mla.decode_plan(4, 128, 64, 1)[0] == 1
    assert f(sl, 4, 128, 64, 1, ws, 256, None) == 0


def test_append_absorb_q_validation_before_launch(lib):
    """mla_append_absorb_q checks the arguments of both calls it stands for, and its workspace
    is the larger of theirs; every call below returns before anything is launched."""
    from mla_latent_kv_13_gb300 import mla
    f = lib.mla_append_absorb_q
    vp, i, fl, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
    f.argtypes = [vp, i, i, vp, vp, vp, i, vp, i, vp, i, vp, vp, vp, i, fl, vp, sz, vp, vp, vp]
    f.restype = ctypes.c_int
    p = 1 << 20  # a 256-byte-aligned stand-in address, never dereferenced
    need = mla.append_absorb_q_workspace_size(128, 7168, 1536, 128)
    assert need >= max(mla.append_kv_workspace_size(128, 7168),
                       mla.absorb_q_workspace_size(128, 7168, 1536, 128))
    ok = [p, 128, 7168, p, p, p, 64, p, 1024, p, 1536, p, p, p, 128, 10000.0, p, need, p, p, None]

    def call(**kw):
        a = list(ok)
        names = ["h", "B", "dm", "w_dkr", "pos", "bt", "maxb", "cache", "nblk", "w_dq", "ql",
                 "w_uq", "w_qr", "w_uk", "H", "theta", "ws", "ws_bytes", "q_lat", "q_rope"]
        for k, v in kw.items():
            a[names.index(k)] = v
        return f(*a)

    assert call(h=None) == 1
    assert call(cache=None) == 1
    assert call(B=0) == 1
    assert call(dm=7000) == 1
    assert call(ql=1500) == 1
    assert call(maxb=0) == 1
    assert call(theta=0.0) == 1
    assert call(H=48) == 2
    assert call(cache=p + 8) == 1     # the cache must be 16-byte aligned
    assert call(ws=p + 16) == 1       # the workspace 256-byte aligned
    assert call(ws_bytes=need - 1) == 3


def test_multi_query_validation_before_launch(lib):
    from mla_latent_kv_13_gb300 import mla
    # s_q * H rows must fit the 128 TMEM lanes; H itself a supported head count
    assert mla.decode_mq_workspace_size(4, 2, 64, 256) > 0
    sz = ctypes.c_size_t(0)
    assert lib.mla_decode_mq_workspace_size(4, 2, 128, 256, 0, ctypes.byref(sz)) == 2
    assert lib.mla_decode_mq_workspace_size(4, 3, 48, 256, 0, ctypes.byref(sz)) == 2
    assert lib.mla_decode_mq_workspace_size(4, 0, 16, 256, 0, ctypes.byref(sz)) == 1
    # s_q = 1 sizes exactly like plain decode
    assert mla.decode_mq_workspace_size(8, 1, 128, 4096, 3) == \
        mla.decode_workspace_size(8, 128, 4096, 3)
    null = ctypes.c_void_p(0)
    lib.mla_decode_attention_mq.restype = ctypes.c_int
    rc = lib.mla_decode_attention_mq(null, null, null, 1, null, 1, null, 1, 2, 16, 64,
                                     ctypes.c_float(0.07), 0, null, ctypes.c_size_t(0), null,
                                     null, null)
    assert rc == 1


def test_selftest_validation_before_launch(lib):
    null = ctypes.c_void_p(0)
    lib.mla_selftest_wait_timeout.restype = ctypes.c_int
    assert lib.mla_selftest_wait_timeout(ctypes.c_uint(0), null, ctypes.c_size_t(256), null) == 1
    assert lib.mla_selftest_wait_timeout(ctypes.c_uint(100), null, ctypes.c_size_t(256), null) == 1


def test_prefill_validation_before_launch(lib):
    from mla_latent_kv_13_gb300 import mla
    assert mla.prefill_workspace_size(128, 0, 4096) > 4096 * 128 * 256 * 2
    sz = ctypes.c_size_t(0)
    assert lib.mla_prefill_workspace_size(48, 0, 64, ctypes.byref(sz)) == 2
    assert lib.mla_prefill_workspace_size(16, -1, 64, ctypes.byref(sz)) == 1
    assert lib.mla_prefill_workspace_size(16, 0, 0, ctypes.byref(sz)) == 1


def _check_schedule(seqlens, max_blocks, clusters, seg_cost=12):
    """Invariants of the balanced schedule (host arithmetic shared with the device)."""
    import numpy as np
    from mla_latent_kv_13_gb300 import mla
    segs, parts = mla.decode_schedule(seqlens, max_blocks, clusters)
    tiles = [(min(max(int(L), 0), 64 * max_blocks) + 63) // 64 for L in seqlens]
    W = sum(v + seg_cost for v in tiles if v > 0)
    P = min(clusters, W)
    covered = [np.zeros(v, dtype=np.int32) for v in tiles]
    by_cluster, parts_of = {}, {}
    for cl, b, t0, t1, part in segs:
        assert 0 <= cl < P and 0 <= t0 < t1 <= tiles[b]
        covered[b][t0:t1] += 1
        by_cluster.setdefault(cl, []).append((b, t0, t1))
        if part < 0:
            assert (t0, t1) == (0, tiles[b])  # written directly: the whole sequence
        else:
            parts_of.setdefault(b, []).append((cl, part))
    for c in covered:  # every tile of every sequence exactly once
        assert (c == 1).all()
    # a cluster's segments run in sequence order; only its first and last may be cut
    for cl, ss in by_cluster.items():
        assert [s[0] for s in ss] == sorted(s[0] for s in ss)
        for k, (b, t0, t1) in enumerate(ss):
            if 0 < k < len(ss) - 1:
                assert (t0, t1) == (0, tiles[b])
    # the parts of a cut sequence: consecutive clusters, consecutive indices in token order
    idx = sorted(p for ps in parts_of.values() for _, p in ps)
    assert idx == list(range(parts)) and parts <= 2 * max(P, 1)
    for b, ps in parts_of.items():
        assert len(ps) >= 2
        cls = [c for c, _ in ps]
        assert cls == list(range(cls[0], cls[0] + len(ps)))
        assert [p for _, p in ps] == list(range(ps[0][1], ps[0][1] + len(ps)))
    # the merge kernel takes one job per cluster, the sequence whose first part that cluster
    # holds: no two cut sequences start in the same cluster
    firsts = [ps[0][0] for ps in parts_of.values()]
    assert len(firsts) == len(set(firsts))
    # balance: no cluster costs more than its share of the weight plus one start-up
    share = -(-W // P) if P else 0
    for ss in by_cluster.values():
        assert sum(seg_cost + t1 - t0 for _, t0, t1 in ss) <= share + seg_cost
    return segs, parts, by_cluster


def test_balanced_schedule_covers_every_tile_once(lib):
    import numpy as np
    from mla_latent_kv_13_gb300 import synth
    rng = np.random.default_rng(5)
    cases = [
        (synth.draw_seqlens(synth.WORKLOADS["mixed"]), 128, 76),   # lengths 1024..8192
        (np.full(128, 8192), 128, 76),                             # equal lengths
        (np.full(76, 8192), 128, 76),
        ([0, 0, 64, 0, 1, 4096, 0], 64, 76),                       # empties, fewer tiles than units
        ([100, 5000, 0, 70000, 1, 65, 640], 1200, 13),             # one dominant sequence
        (rng.integers(0, 3000, 1000), 47, 152),                    # many short ones
        ([8192], 128, 1),
        ([0, 0, 0], 4, 76),                                        # nothing to do
        ([-5, 10 ** 6, 128], 4, 3),                                # clamped like the device
    ]
    for seqlens, mb, clusters in cases:
        _check_schedule(np.asarray(seqlens, dtype=np.int32), mb, clusters)


def test_balanced_schedule_weights_segment_starts(lib):
    """A unit that starts several short sequences gets fewer tiles than one that streams a
    long one: on the mixed-length batch no unit carries more than its share of tiles plus
    start-ups, where equal tile counts would give units of 2 and 5 segments alike."""
    import numpy as np
    from mla_latent_kv_13_gb300 import mla, synth
    seqlens = synth.draw_seqlens(synth.WORKLOADS["mixed"])
    segs, parts, by_cluster = _check_schedule(seqlens, 128, 76)
    tiles = {cl: sum(t1 - t0 for _, t0, t1 in ss) for cl, ss in by_cluster.items()}
    nseg = {cl: len(ss) for cl, ss in by_cluster.items()}
    few = [tiles[c] for c in tiles if nseg[c] == min(nseg.values())]
    many = [tiles[c] for c in tiles if nseg[c] == max(nseg.values())]
    assert min(few) > max(many)
    with pytest.raises(mla.MLAError):
        mla.decode_schedule(seqlens, 128, 0)
    n = ctypes.c_int(0)
    assert lib.mla_decode_schedule(None, 4, 4, 4, None, 0, ctypes.byref(n), None) == 1
    sl = (ctypes.c_int32 * 2)(64, 64)
    assert lib.mla_decode_schedule(sl, 2, 4, 4, None, 0, ctypes.byref(n), None) == 0
    assert n.value >= 1
    assert lib.mla_decode_schedule(sl, 2, 4, 4, None, 3, ctypes.byref(n), None) == 1
