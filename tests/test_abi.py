"""The C-ABI library: it loads, exports what include/diffattn.h declares, and
its host-side validation answers without touching a GPU."""
import ctypes

import pytest

import oracle
from differential_attention_attn_gb300 import build as libbuild
from differential_attention_attn_gb300 import ops


@pytest.fixture(scope="module")
def lib():
    libbuild.build()
    return ops.load()


EXPECTED_ENTRY_POINTS = {
    "diffattn_fwd", "diffattn_fwd_host", "diffattn_fwd_host_staging_bytes",
    "diffattn_fwd_strided", "diffattn_fwd_kv_plan", "diffattn_fwd_kv",
    "diffattn_fwd_kv_strided",
    "diffattn_fwd_kv_noalloc", "diffattn_train_sizes", "diffattn_fwd_train", "diffattn_bwd",
    "diffattn_fwd_train_strided", "diffattn_bwd_strided",
    "diffattn_headnorm", "diffattn_selftest_wait", "diffattn_lambda_init", "diffattn_strerror",
    "diffattn_version"}


def test_exports_every_declared_symbol(lib):
    names = ops.declared_symbols()
    assert set(names) == EXPECTED_ENTRY_POINTS
    for n in names:
        assert hasattr(lib, n), f"{n} declared in include/diffattn.h but not exported"


def test_exports_nothing_undeclared():
    """Every exported diffattn_* function is declared in the header (nm on the built
    library; no compute call)."""
    import subprocess
    lib_path = libbuild.build()
    out = subprocess.run(["nm", "-D", "--defined-only", lib_path], capture_output=True,
                         text=True, check=True).stdout
    exported = {ln.split()[-1] for ln in out.splitlines()
                if ln.split() and ln.split()[-1].startswith("diffattn_") and " T " in ln}
    assert exported == EXPECTED_ENTRY_POINTS


def test_desc_layout_matches_header():
    # int64 x3, int32 x4, float x2, pointer: 56 bytes on LP64.
    assert ctypes.sizeof(ops.Desc) == 56
    assert ops.Desc.status_dev.offset == 48


def test_strerror_and_version(lib):
    for code in range(5):
        assert isinstance(ops.strerror(code), str) and ops.strerror(code)
    assert ops.strerror(99) == "unknown status"
    assert lib.diffattn_version() >= 100


@pytest.mark.parametrize("layer", [1, 2, 5, 12, 24, 100])
def test_lambda_init_matches_oracle(lib, layer):
    assert ops.lambda_init(layer) == pytest.approx(oracle.lambda_init(layer), abs=1e-15)


FAKE = 0x10000  # never dereferenced: validation rejects or returns before any launch


def _call(lib, desc, ptrs=None, lam=FAKE, out=FAKE):
    p = [FAKE] * 5 if ptrs is None else ptrs
    return lib.diffattn_fwd(ctypes.byref(desc) if desc is not None else None,
                            *[ctypes.c_void_p(x) if x else None for x in p],
                            ctypes.c_void_p(lam) if lam else None, None,
                            ctypes.c_void_p(out) if out else None, None)


def test_null_desc_and_pointers(lib):
    assert _call(lib, None) == ops.ERR_INVALID_ARG
    d = ops.make_desc(1, 2, 256, 64, ops.BF16, True, True, 1e-5, 0.2)
    assert _call(lib, d, ptrs=[FAKE, 0, FAKE, FAKE, FAKE]) == ops.ERR_INVALID_ARG
    assert _call(lib, d, lam=0) == ops.ERR_INVALID_ARG
    assert _call(lib, d, out=0) == ops.ERR_INVALID_ARG


@pytest.mark.parametrize("field,value", [("B", -1), ("H", -2), ("N", -5), ("d", 0),
                                         ("dtype", 7), ("eps", -1.0), ("eps", float("nan")),
                                         ("lambda_init", float("inf"))])
def test_invalid_fields(lib, field, value):
    d = ops.make_desc(1, 2, 256, 64, ops.BF16, True, True, 1e-5, 0.2)
    setattr(d, field, value)
    assert _call(lib, d) == ops.ERR_INVALID_ARG


def test_empty_problem_is_ok_without_launch(lib):
    for B, H, N in ((0, 4, 128), (2, 0, 128), (1, 4, 0)):
        d = ops.make_desc(B, H, N, 64, ops.BF16, True, True, 1e-5, 0.2)
        assert _call(lib, d, ptrs=[0] * 5, lam=0, out=0) == ops.OK


def test_bf16_domain(lib):
    d = ops.make_desc(1, 2, 256, 96, ops.BF16, True, True, 1e-5, 0.2)  # d = 64 and 128 only
    assert _call(lib, d) == ops.ERR_UNSUPPORTED
    d = ops.make_desc(1, 2, 256, 64, ops.BF16, True, True, 1e-5, 0.2)
    assert _call(lib, d, ptrs=[FAKE + 8] + [FAKE] * 4) == ops.ERR_INVALID_ARG
    assert _call(lib, d, out=FAKE + 2) == ops.ERR_INVALID_ARG


def test_f32_domain(lib):
    d = ops.make_desc(1, 1, 5000, 8, ops.F32, False, False, 1e-5, 0.0)
    assert _call(lib, d) == ops.ERR_UNSUPPORTED
    d = ops.make_desc(1, 1, 16, 129, ops.F32, False, False, 1e-5, 0.0)
    assert _call(lib, d) == ops.ERR_UNSUPPORTED


def test_headnorm_validation(lib):
    d = ops.make_desc(1, 1, 16, 200, ops.F32, False, True, 1e-5, 0.0)
    assert lib.diffattn_headnorm(ctypes.byref(d), ctypes.c_void_p(FAKE), None,
                                 ctypes.c_void_p(FAKE), None) == ops.ERR_UNSUPPORTED
    d = ops.make_desc(1, 1, 16, 8, ops.F32, False, True, 1e-5, 0.0)
    assert lib.diffattn_headnorm(ctypes.byref(d), None, None, ctypes.c_void_p(FAKE),
                                 None) == ops.ERR_INVALID_ARG


# ----------------------------------------------------------------------------- fwd_kv
PART_FLOATS = 2 * (128 * 128 + 2 * 128)  # per (work item, split): two maps' O, m and l


def _plan(lib, desc, n_kv, splits):
    sp, nb = ctypes.c_int(-1), ctypes.c_size_t(0)
    st = lib.diffattn_fwd_kv_plan(ctypes.byref(desc), n_kv, splits, ctypes.byref(sp),
                                  ctypes.byref(nb))
    return st, sp.value, nb.value


def _call_kv(lib, desc, n_kv, splits, ws=FAKE, ws_bytes=1 << 40):
    p = [ctypes.c_void_p(FAKE)] * 5
    return lib.diffattn_fwd_kv(ctypes.byref(desc), n_kv, *p, ctypes.c_void_p(FAKE), None,
                               ctypes.c_void_p(FAKE), splits,
                               ctypes.c_void_p(ws) if ws else None, ws_bytes, None)


def test_kv_plan_explicit_splits(lib):
    d = ops.make_desc(1, 4, 512, 64, ops.BF16, True, True, 1e-5, 0.2)
    assert _plan(lib, d, 512, 3) == (ops.OK, 3, 16 * 3 * PART_FLOATS * 4)
    assert _plan(lib, d, 512, 1) == (ops.OK, 1, 0)
    assert _plan(lib, d, 512, 100) == (ops.OK, 4, 16 * 4 * PART_FLOATS * 4)  # 4 key tiles
    dec = ops.make_desc(2, 8, 1, 64, ops.BF16, True, True, 1e-5, 0.2)  # decoding: one query
    assert _plan(lib, dec, 16384, 8) == (ops.OK, 8, 16 * 8 * PART_FLOATS * 4)
    empty = ops.make_desc(0, 8, 1, 64, ops.BF16, True, True, 1e-5, 0.2)
    assert _plan(lib, empty, 100, 0) == (ops.OK, 1, 0)


def test_kv_validation(lib):
    d = ops.make_desc(1, 4, 512, 64, ops.BF16, True, True, 1e-5, 0.2)
    assert _plan(lib, d, 511, 1)[0] == ops.ERR_INVALID_ARG       # causal, fewer keys than queries
    assert _plan(lib, d, -1, 1)[0] == ops.ERR_INVALID_ARG
    assert _plan(lib, d, 512, -1)[0] == ops.ERR_INVALID_ARG
    assert _plan(lib, d, 512, 257)[0] == ops.ERR_INVALID_ARG
    nc = ops.make_desc(1, 4, 512, 64, ops.BF16, False, True, 1e-5, 0.2)
    assert _plan(lib, nc, 0, 1)[0] == ops.ERR_INVALID_ARG        # softmax over no keys
    assert _plan(lib, nc, 100, 1)[0] == ops.OK                    # fewer keys is fine unmasked
    f32 = ops.make_desc(1, 4, 64, 8, ops.F32, True, True, 1e-5, 0.2)
    assert _plan(lib, f32, 64, 1)[0] == ops.ERR_UNSUPPORTED
    wide = ops.make_desc(1, 4, 64, 128, ops.BF16, True, True, 1e-5, 0.2)
    assert _plan(lib, wide, 64, 1)[:2] == (ops.OK, 1)             # d = 128: single pass
    assert _plan(lib, wide, 4096, 0)[:2] == (ops.OK, 1)           # the library picks 1
    assert _plan(lib, wide, 4096, 2)[0] == ops.ERR_UNSUPPORTED    # no split-KV at d = 128
    wide8 = ops.make_desc(1, 4, 64, 128, ops.E4M3_QK, True, True, 1e-5, 0.2)
    assert _plan(lib, wide8, 64, 1)[0] == ops.ERR_UNSUPPORTED
    odd = ops.make_desc(1, 4, 64, 96, ops.BF16, True, True, 1e-5, 0.2)
    assert _plan(lib, odd, 64, 1)[0] == ops.ERR_UNSUPPORTED
    assert lib.diffattn_fwd_kv_plan(ctypes.byref(d), 512, 1, None, None) == ops.ERR_INVALID_ARG
    # split launches need a large enough, aligned workspace (checked before any launch)
    assert _call_kv(lib, d, 512, 2, ws=0) == ops.ERR_INVALID_ARG
    assert _call_kv(lib, d, 512, 2, ws_bytes=16 * 2 * PART_FLOATS * 4 - 4) == ops.ERR_INVALID_ARG
    assert _call_kv(lib, d, 512, 2, ws=FAKE + 4) == ops.ERR_INVALID_ARG
    assert _call_kv(lib, d, 511, 1) == ops.ERR_INVALID_ARG


# ----------------------------------------------------------------------------- training
def test_train_sizes(lib):
    B, H, N = 2, 3, 300
    d = ops.make_desc(B, H, N, 64, ops.BF16, True, True, 1e-5, 0.2)
    a, b = ctypes.c_size_t(0), ctypes.c_size_t(0)
    assert lib.diffattn_train_sizes(ctypes.byref(d), ctypes.byref(a), ctypes.byref(b)) == ops.OK
    n_pad = 384
    assert a.value == 4 * (2 * B * H * N * 128 + 2 * B * H * n_pad)
    assert b.value >= 4 * (B * H * N * 64 + 2 * B * H * n_pad + 2 * B * H * N * 64 + B * H * N * 128)
    f32 = ops.make_desc(B, H, N, 8, ops.F32, True, True, 1e-5, 0.2)
    assert lib.diffattn_train_sizes(ctypes.byref(f32), ctypes.byref(a),
                                    ctypes.byref(b)) == ops.ERR_UNSUPPORTED
    # d = 128: fp32 map outputs [2][BH][N][256] and fp32 log2-sum-exp, each region
    # rounded to 256 bytes; the workspace holds dO, c D and the fp32 dq accumulator
    r256 = lambda x: (x + 255) // 256 * 256
    wide = ops.make_desc(B, H, N, 128, ops.BF16, True, True, 1e-5, 0.2)
    assert lib.diffattn_train_sizes(ctypes.byref(wide), ctypes.byref(a), ctypes.byref(b)) == ops.OK
    assert a.value == r256(2 * B * H * N * 256 * 4) + r256(2 * B * H * n_pad * 4)
    assert b.value == (r256(B * H * N * 256 * 2) + r256(2 * B * H * n_pad * 4) +
                       r256(2 * B * H * N * 128 * 4))
    odd = ops.make_desc(B, H, N, 96, ops.BF16, True, True, 1e-5, 0.2)
    assert lib.diffattn_train_sizes(ctypes.byref(odd), ctypes.byref(a),
                                    ctypes.byref(b)) == ops.ERR_UNSUPPORTED


@pytest.mark.parametrize("dh", [64, 128])
def test_bwd_validation_before_launch(lib, dh):
    d = ops.make_desc(1, 2, 256, dh, ops.BF16, True, True, 1e-5, 0.2)
    f = ctypes.c_void_p(FAKE)
    # q1 k1 q2 k2 v | lambda norm_w saved dy | dq1 dk1 dq2 dk2 dv | dlambda dnorm_w
    args = [f] * 5 + [f, None, f, f] + [f] * 5 + [f, None]
    # workspace too small
    assert lib.diffattn_bwd(ctypes.byref(d), *args, f, 16, None) == ops.ERR_INVALID_ARG
    # workspace not 256-byte aligned
    assert lib.diffattn_bwd(ctypes.byref(d), *args, ctypes.c_void_p(FAKE + 16), 1 << 40,
                            None) == ops.ERR_INVALID_ARG
    # missing dy
    bad = list(args)
    bad[8] = None
    assert lib.diffattn_bwd(ctypes.byref(d), *bad, f, 1 << 40, None) == ops.ERR_INVALID_ARG
    # fwd_train needs the saved buffer, large enough and aligned
    assert lib.diffattn_fwd_train(ctypes.byref(d), *[f] * 5, f, None, f, None, 1 << 40,
                                  None) == ops.ERR_INVALID_ARG
    saved, ws = ctypes.c_size_t(0), ctypes.c_size_t(0)
    assert lib.diffattn_train_sizes(ctypes.byref(d), ctypes.byref(saved),
                                    ctypes.byref(ws)) == ops.OK
    assert lib.diffattn_fwd_train(ctypes.byref(d), *[f] * 5, f, None, f, f, saved.value - 1,
                                  None) == ops.ERR_INVALID_ARG
    assert lib.diffattn_fwd_train(ctypes.byref(d), *[f] * 5, f, None, f,
                                  ctypes.c_void_p(FAKE + 8), saved.value,
                                  None) == ops.ERR_INVALID_ARG
    # the backward's workspace one byte short
    assert lib.diffattn_bwd(ctypes.byref(d), *args, f, ws.value - 1, None) == ops.ERR_INVALID_ARG
    # a misaligned gradient
    bad = list(args)
    bad[10] = ctypes.c_void_p(FAKE + 4)
    assert lib.diffattn_bwd(ctypes.byref(d), *bad, f, 1 << 40, None) == ops.ERR_INVALID_ARG


def test_headnorm_mode_validation(lib):
    d = ops.make_desc(1, 2, 256, 64, ops.BF16, True, 3, 1e-5, 0.2)
    assert _call(lib, d) == ops.ERR_INVALID_ARG
    # the group form is trainable: same buffer sizes as the RMS form
    g = ops.make_desc(1, 2, 256, 64, ops.BF16, True, 2, 1e-5, 0.2)
    r = ops.make_desc(1, 2, 256, 64, ops.BF16, True, 1, 1e-5, 0.2)
    a, b = ctypes.c_size_t(0), ctypes.c_size_t(0)
    a1, b1 = ctypes.c_size_t(0), ctypes.c_size_t(0)
    assert lib.diffattn_train_sizes(ctypes.byref(g), ctypes.byref(a), ctypes.byref(b)) == ops.OK
    assert lib.diffattn_train_sizes(ctypes.byref(r), ctypes.byref(a1), ctypes.byref(b1)) == ops.OK
    assert (a.value, b.value) == (a1.value, b1.value) and a.value > 0


def test_strided_validation_before_launch(lib):
    d = ops.make_desc(1, 2, 256, 64, ops.BF16, True, 1, 1e-5, 0.2)
    f = ctypes.c_void_p(FAKE)
    good = [ops.Strides(2 * 256 * 64, 256 * 64, 64)] * 4 + [ops.Strides(2 * 256 * 128, 256 * 128, 128)] * 2
    for bad in (ops.Strides(0, 64, 64), ops.Strides(8, 12, 64), ops.Strides(8, 8, 1 << 40)):
        arr = (ops.Strides * 6)(*(good[:2] + [bad] + good[3:]))
        assert lib.diffattn_fwd_strided(ctypes.byref(d), f, f, f, f, f, f, None, f, arr,
                                        None) == ops.ERR_INVALID_ARG
    assert lib.diffattn_fwd_strided(ctypes.byref(d), f, f, f, f, f, f, None, f, None,
                                    None) == ops.ERR_INVALID_ARG
    f32 = ops.make_desc(1, 2, 256, 64, ops.F32, True, 1, 1e-5, 0.2)
    arr = (ops.Strides * 6)(*good)
    assert lib.diffattn_fwd_strided(ctypes.byref(f32), f, f, f, f, f, f, None, f, arr,
                                    None) == ops.ERR_UNSUPPORTED


def test_kv_plan_accepts_e4m3_queries_keys(lib):
    """The key/value-cache entries take DIFFATTN_E4M3_QK (d = 64, headnorm 0 or 1):
    the planner answers as for bf16; the group norm is refused before any launch."""
    bf = ops.make_desc(1, 4, 512, 64, ops.BF16, True, True, 1e-5, 0.2)
    e4 = ops.make_desc(1, 4, 512, 64, ops.E4M3_QK, True, True, 1e-5, 0.2)
    assert _plan(lib, e4, 512, 3) == _plan(lib, bf, 512, 3)
    dec = ops.make_desc(1, 8, 1, 64, ops.E4M3_QK, True, 0, 1e-5, 0.2)
    assert _plan(lib, dec, 16384, 4) == (ops.OK, 4, 8 * 4 * PART_FLOATS * 4)
    grp = ops.make_desc(1, 4, 512, 64, ops.E4M3_QK, True, 2, 1e-5, 0.2)
    assert _plan(lib, grp, 512, 2)[0] == ops.ERR_UNSUPPORTED
    wide = ops.make_desc(1, 4, 512, 128, ops.E4M3_QK, True, True, 1e-5, 0.2)
    assert _plan(lib, wide, 512, 2)[0] == ops.ERR_UNSUPPORTED


def test_strided_domain_takes_both_head_widths(lib):
    """diffattn_fwd_strided serves d = 64 and d = 128; any other width is refused as
    unsupported.  The accepted widths are stopped by a misaligned output pointer, the
    next check, so nothing is ever launched whatever the machine."""
    f = ctypes.c_void_p(FAKE)
    misaligned = ctypes.c_void_p(FAKE + 4)
    for d_half, ok in ((64, True), (128, True), (96, False), (32, False)):
        desc = ops.make_desc(1, 2, 256, d_half, ops.BF16, True, 1, 1e-5, 0.2)
        arr = (ops.Strides * 6)(*([ops.Strides(2 * 256 * d_half, 256 * d_half, d_half)] * 4 +
                                  [ops.Strides(2 * 256 * 2 * d_half, 256 * 2 * d_half,
                                               2 * d_half)] * 2))
        st = lib.diffattn_fwd_strided(ctypes.byref(desc), f, f, f, f, f, f, None, misaligned,
                                      arr, None)
        assert st == (ops.ERR_INVALID_ARG if ok else ops.ERR_UNSUPPORTED), (d_half, st)


def test_debug_build_exports_the_same_entry_points():
    """The bounds-checked variant (DIFFATTN_DEBUG) builds and exports the same C ABI;
    its strerror knows the bounds status (host-only, no GPU)."""
    path = libbuild.build(debug=True)
    dbg = ops.bind(ctypes.CDLL(path))
    for n in EXPECTED_ENTRY_POINTS:
        assert hasattr(dbg, n)
    assert dbg.diffattn_strerror(ops.ERR_BOUNDS).decode() == "kernel bounds check failed (debug build)"


def test_fwd_host_staging_and_validation(lib):
    """diffattn_fwd_host: staging size (five inputs and the output, each rounded up
    to 256 bytes) and argument checks that return before any copy is queued."""
    B, H, N = 2, 3, 300
    d = ops.make_desc(B, H, N, 64, ops.BF16, True, True, 1e-5, 0.2)
    n = ctypes.c_size_t(0)
    assert lib.diffattn_fwd_host_staging_bytes(ctypes.byref(d), ctypes.byref(n)) == ops.OK
    r = lambda x: (x + 255) // 256 * 256
    qk, wide = B * H * N * 64 * 2, B * H * N * 128 * 2
    assert n.value == 4 * r(qk) + 2 * r(wide)
    f32 = ops.make_desc(1, 1, 6, 8, ops.F32, False, False, 1e-5, 0.2)
    assert lib.diffattn_fwd_host_staging_bytes(ctypes.byref(f32), ctypes.byref(n)) == ops.OK
    assert n.value == 4 * r(6 * 8 * 4) + 2 * r(6 * 16 * 4)
    assert lib.diffattn_fwd_host_staging_bytes(ctypes.byref(d), None) == ops.ERR_INVALID_ARG
    assert lib.diffattn_fwd_host_staging_bytes(None, ctypes.byref(n)) == ops.ERR_INVALID_ARG
    need = 4 * r(qk) + 2 * r(wide)
    f = ctypes.c_void_p(FAKE)
    args = [f] * 5 + [f, None, f]
    # NULL, misaligned, short staging
    assert lib.diffattn_fwd_host(ctypes.byref(d), *args, None, need, None) == ops.ERR_INVALID_ARG
    assert lib.diffattn_fwd_host(ctypes.byref(d), *args, ctypes.c_void_p(FAKE + 16), need,
                                 None) == ops.ERR_INVALID_ARG
    assert lib.diffattn_fwd_host(ctypes.byref(d), *args, f, need - 1, None) == ops.ERR_INVALID_ARG
    # NULL host input or output
    assert lib.diffattn_fwd_host(ctypes.byref(d), None, *args[1:], f, need,
                                 None) == ops.ERR_INVALID_ARG
    assert lib.diffattn_fwd_host(ctypes.byref(d), *args[:7], None, f, need,
                                 None) == ops.ERR_INVALID_ARG
    # empty problem: nothing to do
    e = ops.make_desc(0, 3, 300, 64, ops.BF16, True, True, 1e-5, 0.2)
    assert lib.diffattn_fwd_host(ctypes.byref(e), *args, None, 0, None) == ops.OK


def test_strided_training_validation_before_launch(lib):
    """diffattn_fwd_train_strided / diffattn_bwd_strided: missing or bad strides and
    unsupported dtypes or widths are refused before anything is launched."""
    d = ops.make_desc(1, 2, 256, 64, ops.BF16, True, 1, 1e-5, 0.2)
    f = ctypes.c_void_p(FAKE)
    s64 = ops.Strides(2 * 256 * 64, 256 * 64, 64)
    s128 = ops.Strides(2 * 256 * 128, 256 * 128, 128)
    fwd_good = [s64] * 4 + [s128] * 2
    assert lib.diffattn_fwd_train_strided(ctypes.byref(d), *[f] * 5, f, None, f, f, 1 << 40,
                                          None, None) == ops.ERR_INVALID_ARG
    arr = (ops.Strides * 6)(*(fwd_good[:4] + [ops.Strides(8, 8, 12)] + fwd_good[5:]))
    assert lib.diffattn_fwd_train_strided(ctypes.byref(d), *[f] * 5, f, None, f, f, 1 << 40,
                                          arr, None) == ops.ERR_INVALID_ARG
    for dt, dh in ((ops.F32, 64), (ops.BF16, 96)):
        other = ops.make_desc(1, 2, 256, dh, dt, True, 1, 1e-5, 0.2)
        arr = (ops.Strides * 6)(*fwd_good)
        assert lib.diffattn_fwd_train_strided(ctypes.byref(other), *[f] * 5, f, None, f, f,
                                              1 << 40, arr, None) == ops.ERR_UNSUPPORTED
    # q1 k1 q2 k2 v | lambda norm_w saved dy | dq1 dk1 dq2 dk2 dv | dlambda dnorm_w
    args = [f] * 5 + [f, None, f, f] + [f] * 5 + [f, None]
    bwd_good = [s64] * 4 + [s128] * 2 + [s64] * 4 + [s128]
    assert lib.diffattn_bwd_strided(ctypes.byref(d), *args, f, 1 << 40, None,
                                    None) == ops.ERR_INVALID_ARG
    for i in range(11):  # a bad stride in any of the eleven positions
        bad = list(bwd_good)
        bad[i] = ops.Strides(bad[i].b, 0, bad[i].n)
        arr = (ops.Strides * 11)(*bad)
        assert lib.diffattn_bwd_strided(ctypes.byref(d), *args, f, 1 << 40, arr,
                                        None) == ops.ERR_INVALID_ARG, i
    arr = (ops.Strides * 11)(*bwd_good)
    assert lib.diffattn_bwd_strided(ctypes.byref(d), *args, f, 16, arr,
                                    None) == ops.ERR_INVALID_ARG  # short workspace
