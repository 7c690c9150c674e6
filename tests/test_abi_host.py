"""The C-ABI library loads, exports every declared entry point, sizes its
workspace and rejects invalid arguments on the host before any launch.
No GPU is needed: every call here fails validation before touching CUDA."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def L():
    import __graft_entry__ as g
    g.build()
    import sparse_kv_verify_gb300 as dk
    return dk


def declared_functions():
    src = open(os.path.join(ROOT, "include", "dustin.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?\w+\s*\*?\s*(\w+)\s*\(", src, flags=re.M)))


def test_exports_every_declared_symbol(L):
    names = declared_functions()
    assert len(names) >= 10
    lib = L.lib()
    for n in names:
        assert hasattr(lib, n), n
    assert set(L.EXPORTS) <= set(names)


def test_version(L):
    assert "sm_103a" in L.version()


def _fake_kv(L, hkv=8, d=128, Lcap=1024, ptr=0x10000):
    return L.binding.CKV(ptr, hkv, d, Lcap * d * hkv, Lcap * d, d) if hasattr(L, "binding") else None


def test_workspace_sizing(L):
    from sparse_kv_verify_gb300 import binding as bd
    p = bd.CParams(2, 1024, 4, 4, 32, 32, 128)
    lib = L.lib()
    base = 256 + 65536          # error word + selection arrival counters

    def r256(x):
        return (x + 255) // 256 * 256

    # selection scratch, B = 2, Lcap = 1024: histograms [B][2][4096] int32
    # and the general path's bitmaps [B][(Lcap + 127) / 32 + 2] words
    sel = r256(2 * 2 * 4096 * 4) + r256(2 * (1151 // 32 + 2) * 4)
    assert lib.dustin_workspace_bytes(ctypes.byref(p), None, None, None, 0, 0, 0, 0, 0) == base + sel
    kv_t = (bd.CKV * 1)(bd.CKV(0x10000, 2, 128, 2 * 1024 * 128, 1024 * 128, 128))
    kv_d = (bd.CKV * 1)(bd.CKV(0x20000, 1, 64, 1024 * 64, 1024 * 64, 64))
    qt = (ctypes.c_void_p * 1)(0x30000)
    qd = (ctypes.c_void_p * 1)(0x40000)
    tgt = bd.CSignal(1, 8, 5, qt, kv_t)
    dft = bd.CSignal(1, 2, 4, qd, kv_d)
    srh = (bd.CSRH * 3)(bd.CSRH(1, 0, 0), bd.CSRH(1, 0, 7), bd.CSRH(0, 0, 1))
    n = lib.dustin_workspace_bytes(ctypes.byref(p), ctypes.byref(dft), ctypes.byref(tgt), srh, 3,
                                   0, 0, 0, 0)
    # logits of 3 slabs (target heads 0 and 7 sit in different KV groups):
    # (5 + 5 + 4 pairs) x B x Lcap fp32, plus per-segment statistics
    assert n > base + (5 + 5 + 4) * 2 * 1024 * 4
    # verification adds per-unit partial slots [units][max_seg][NQ][d + 2]
    nv = lib.dustin_workspace_bytes(ctypes.byref(p), None, None, None, 0, 8, 2, 128, 1)
    assert nv > base
    assert lib.dustin_workspace_bytes(ctypes.byref(p), None, None, None, 0, 8, 3, 128, 1) == 0
    assert lib.dustin_workspace_bytes(ctypes.byref(p), None, None, None, 0, 8, 2, 96, 1) == 0
    assert lib.dustin_workspace_bytes(ctypes.byref(p), None, None, None, 0, 8, 2, 128, 17) == 0
    # the draft block is at most 64 rows (gamma + 1 <= 64), whatever the group size
    p64 = bd.CParams(2, 1024, 63, 4, 32, 32, 128)
    p65 = bd.CParams(2, 1024, 64, 4, 32, 32, 128)
    assert lib.dustin_workspace_bytes(ctypes.byref(p64), None, None, None, 0, 8, 8, 128, 1) > base
    assert lib.dustin_workspace_bytes(ctypes.byref(p65), None, None, None, 0, 8, 8, 128, 1) == 0
    # duplicate SRH, bad channel, head out of range -> 0 (invalid)
    for bad in [(1, 0, 0), ]:
        srh2 = (bd.CSRH * 2)(bd.CSRH(1, 0, 0), bd.CSRH(*bad))
        assert lib.dustin_workspace_bytes(ctypes.byref(p), ctypes.byref(dft), ctypes.byref(tgt), srh2, 2,
                                          0, 0, 0, 0) == 0
    for bad in [(2, 0, 0), (1, 0, 8), (1, 1, 0), (0, 0, 2)]:
        srh2 = (bd.CSRH * 1)(bd.CSRH(*bad))
        assert lib.dustin_workspace_bytes(ctypes.byref(p), ctypes.byref(dft), ctypes.byref(tgt), srh2, 1,
                                          0, 0, 0, 0) == 0


def test_invalid_params_rejected(L):
    from sparse_kv_verify_gb300 import binding as bd
    lib = L.lib()
    ws = 0x100000   # never dereferenced: validation fails first
    good = dict(B=2, Lcap=1024, gamma=4, sinks=4, window=32, m=32, k=128)
    bads = [dict(B=0), dict(Lcap=0), dict(Lcap=(1 << 20) + 1), dict(k=0), dict(gamma=-1),
            dict(sinks=100, window=100), dict(m=-1)]
    for over in bads:
        d = dict(good)
        d.update(over)
        p = bd.CParams(*[d[f] for f in ("B", "Lcap", "gamma", "sinks", "window", "m", "k")])
        assert lib.dustin_select(ctypes.byref(p), 0x1000, 0x2000, 0x3000, ws, 1 << 20, None) == -1
        assert lib.dustin_workspace_bytes(ctypes.byref(p), None, None, None, 0, 0, 0, 0, 0) == 0
    p = bd.CParams(*good.values())
    assert lib.dustin_select(ctypes.byref(p), None, 0x2000, 0x3000, ws, 1 << 20, None) == -1
    assert lib.dustin_select(ctypes.byref(p), 0x1000, 0x2000, 0x3000, None, 1 << 20, None) == -5
    assert lib.dustin_select(ctypes.byref(p), 0x1000, 0x2000, 0x3000, ws + 8, 1 << 20, None) == -5
    assert lib.dustin_select(ctypes.byref(p), 0x1000, 0x2000, 0x3000, ws, 16, None) == -5


def test_invalid_verify_arguments_rejected(L):
    from sparse_kv_verify_gb300 import binding as bd
    lib = L.lib()
    p = bd.CParams(2, 1024, 4, 4, 32, 32, 128)
    k = bd.CKV(0x10000, 8, 128, 8 * 1024 * 128, 1024 * 128, 128)
    ws = 0x100000
    args = lambda **o: dict(dict(hq=64, q=0x1000, k=k, v=k, kb=0x2000, vb=0x3000, i=0x4000,
                                 sl=0x5000, o=0x6000), **o)

    def call(a):
        return lib.dustin_verify_attn(ctypes.byref(p), a["hq"], a["q"], a["k"], a["v"], a["kb"],
                                      a["vb"], a["i"], a["sl"], a["o"], ws, 1 << 20, None)
    assert call(args(q=None)) == -1
    assert call(args(q=0x1008)) == -1                      # misaligned
    assert call(args(hq=60)) == -1                         # hq not a multiple of hkv
    assert call(args(k=bd.CKV(0x10000, 8, 96, 0, 0, 96))) == -1   # unsupported head dim
    assert call(args(k=bd.CKV(0x10000, 8, 128, 8 * 1024 * 128, 1024 * 128, 100))) == -1
    assert call(args(v=bd.CKV(0x10000, 4, 128, 4 * 1024 * 128, 1024 * 128, 128))) == -1
    assert call(args(i=None)) == -1
    p2 = bd.CParams(2, 1024, 16, 4, 32, 32, 128)           # 17 x 8 query rows > 128
    assert lib.dustin_verify_attn(ctypes.byref(p2), 64, 0x1000, k, k, 0x2000, 0x3000, 0x4000,
                                  0x5000, 0x6000, ws, 1 << 20, None) == -2
    assert lib.dense_verify_attn(ctypes.byref(p), 64, 0x1000, k, k, 0x2000, 0x3000, None,
                                 0x6000, ws, 1 << 20, None) == -1
    # the draft block is one 64-key tile: gamma + 1 = 65 rows is refused even
    # when the query rows fit (Hq / Hkv = 1)
    k1 = bd.CKV(0x10000, 8, 128, 8 * 1024 * 128, 1024 * 128, 128)
    p64 = bd.CParams(2, 1024, 64, 4, 32, 32, 128)
    assert lib.dustin_verify_attn(ctypes.byref(p64), 8, 0x1000, k1, k1, 0x2000, 0x3000, 0x4000,
                                  0x5000, 0x6000, ws, 1 << 20, None) == -2
    assert lib.dense_verify_attn(ctypes.byref(p64), 8, 0x1000, k1, k1, 0x2000, 0x3000, 0x5000,
                                 0x6000, ws, 1 << 20, None) == -2


def test_invalid_append_arguments_rejected(L):
    from sparse_kv_verify_gb300 import binding as bd
    lib = L.lib()
    p = bd.CParams(2, 1024, 4, 4, 32, 32, 128)
    k = (bd.CKV * 17)(*[bd.CKV(0x10000, 8, 128, 8 * 1024 * 128, 1024 * 128, 128)] * 17)
    kb = (ctypes.c_void_p * 17)(*[0x2000] * 17)
    ws = 0x100000
    assert lib.dustin_kv_append(ctypes.byref(p), 17, k, k, kb, kb, 0x1000, 0x2000, ws, 1 << 20, None) == -2
    assert lib.dustin_kv_append(ctypes.byref(p), 0, k, k, kb, kb, 0x1000, 0x2000, ws, 1 << 20, None) == -1
    assert lib.dustin_kv_append(ctypes.byref(p), 2, k, k, kb, kb, None, 0x2000, ws, 1 << 20, None) == -1
    kb_bad = (ctypes.c_void_p * 2)(0x2000, 0x2004)
    assert lib.dustin_kv_append(ctypes.byref(p), 2, k, k, kb_bad, kb, 0x1000, 0x2000, ws, 1 << 20, None) == -1


def test_compact_refuses_seq_len_c_aliasing_seq_len(L):
    """seq_len_c is written while other CTAs still read seq_len, so the two
    may not be one array; the refusal comes before any launch."""
    from sparse_kv_verify_gb300 import binding as bd
    lib = L.lib()
    p = bd.CParams(2, 1024, 4, 4, 32, 32, 128)
    kv = (bd.CKV * 1)(bd.CKV(0x10000, 8, 128, 8 * 1024 * 128, 1024 * 128, 128))
    kc = (bd.CKV * 1)(bd.CKV(0x20000, 8, 128, 8 * 128 * 128, 128 * 128, 128))
    ws = 0x100000
    assert lib.dustin_compact_kv(ctypes.byref(p), 1, kv, kv, 0x1000, 0x2000, kc, kc, 0x2000,
                                 ws, 1 << 20, None) == -1
    assert lib.dustin_compact_kv(ctypes.byref(p), 1, kv, kv, 0x1000, 0x2000, kc, kc, None,
                                 ws, 1 << 20, None) == -1
    assert lib.dustin_compact_kv(ctypes.byref(p), 1, kv, kv, 0x1000, 0x2000, kc, kc, 0x3000,
                                 None, 1 << 20, None) == -5


def test_wait_selftest_argument_checks(L):
    """The wait limit must lie in [1 us, 1 s]; the output must be a non-null
    8-byte-aligned device pointer; the workspace needs its header."""
    lib = L.lib()
    ws = 0x100000
    assert lib.dustin_wait_selftest(999, 0x2000, ws, 256, None) == -1
    assert lib.dustin_wait_selftest(1000000001, 0x2000, ws, 256, None) == -1
    assert lib.dustin_wait_selftest(1000000, None, ws, 256, None) == -1
    assert lib.dustin_wait_selftest(1000000, 0x2004, ws, 256, None) == -1
    assert lib.dustin_wait_selftest(1000000, 0x2000, None, 256, None) == -5
    assert lib.dustin_wait_selftest(1000000, 0x2000, ws, 128, None) == -5


def test_split_units_matches_brute_force(L):
    """The host's list of units that the verification split cuts across CTAs
    equals a brute-force assignment of every tile to its CTA."""
    from sparse_kv_verify_gb300 import binding as bd
    for (B, hkv, nl, G, tu) in [(2, 8, 1, 152, 33), (16, 8, 1, 152, 33), (1, 1, 1, 5, 7),
                                (3, 2, 2, 5, 4), (4, 8, 8, 152, 65)]:
        p = bd.Params(B, 1024, 4, 4, 32, 32, 128)
        T = B * hkv * nl * tu
        owner = [0] * T
        for c in range(G):
            for t in range(c * T // G, (c + 1) * T // G):
                owner[t] = c
        brute = [u for u in range(B * hkv * nl)
                 if len({owner[t] for t in range(u * tu, (u + 1) * tu)}) > 1]
        assert bd.split_units(p, hkv, nl, G, tu) == brute


def test_step_rejects_null_and_too_many_layers(L):
    from sparse_kv_verify_gb300 import binding as bd
    lib = L.lib()
    assert lib.dustin_verify_step(None, 0x100000, 1 << 20, None) == -1
    assert lib.dustin_check(None, None, None) == -5
    assert lib.dustin_workspace_init(None, 256, None) == -5


def test_step_launch_count(L):
    """The launch-count query plans like dustin_verify_step: two kernels per
    scoring group (stream, normalise), then select, then verify and the merge
    of split units."""
    from sparse_kv_verify_gb300 import binding as bd
    lib = L.lib()

    def step(B, Lcap):
        kv_t = (bd.CKV * 1)(bd.CKV(0x10000, 8, 128, 8 * Lcap * 128, Lcap * 128, 128))
        kv_d = (bd.CKV * 1)(bd.CKV(0x20000, 2, 64, 2 * Lcap * 64, Lcap * 64, 64))
        q = (ctypes.c_void_p * 1)(0x30000)
        tgt = bd.CSignal(1, 64, 6, q, kv_t)
        dft = bd.CSignal(1, 14, 5, q, kv_d)
        srh = (bd.CSRH * 8)(*[bd.CSRH(1, 0, h) for h in (0, 16, 32, 48)],
                            *[bd.CSRH(0, 0, h) for h in (0, 3, 7, 10)])
        lay = (bd.CVerifyLayer * 1)()
        s = bd.CStep(bd.CParams(B, Lcap, 5, 16, 256, 512, 2048), ctypes.pointer(dft),
                     ctypes.pointer(tgt), srh, 8, 64, 1, lay, 0x40000, 0x50000, 0x60000, None)
        n, g = ctypes.c_int32(0), ctypes.c_int32(0)
        st = lib.dustin_step_launches(ctypes.byref(s), ctypes.byref(n), ctypes.byref(g))
        return st, n.value, g.value, (dft, tgt, srh, lay, kv_t, kv_d, q)

    st, n, g, _ = step(2, 4096)
    assert (st, n, g) == (0, 5, 2)              # one group
    # 44 logits rows of 32 K positions per sequence: 5.78 MB; 16 sequences fit
    # the L2 budget in one group, 20 need two, of equal size
    st, n, g, _ = step(16, 32832)
    assert (st, n, g) == (0, 5, 16)
    st, n, g, _ = step(20, 32832)
    assert (st, n, g) == (0, 2 * 2 + 3, 10)
    assert lib.dustin_step_launches(None, ctypes.byref(ctypes.c_int32()),
                                    ctypes.byref(ctypes.c_int32())) == -1
