"""Host-side checks of the C ABI: the library builds and loads, exports every
function include/bitmtp_linear.h declares, and rejects invalid arguments on
the host before any CUDA call.  No kernel is launched: calls that pass
validation are only made where no GPU is present (they must then report
BITMTP_ERR_UNSUPPORTED)."""
import ctypes

import pytest
import torch

import oracle
from ternary_w2a8_linear_gb300 import build, linear as L

FAKE = 0x10000  # 16-byte aligned, never dereferenced


@pytest.fixture(scope="module")
def lib():
    build.build()
    return L.load()


def test_exports_every_header_symbol(lib):
    syms = L.header_symbols()
    assert set(syms) == {
        "bitmtp_linear_packed_bytes", "bitmtp_linear_pack", "bitmtp_linear_quant_act",
        "bitmtp_linear_gemm", "bitmtp_linear_gemm_grouped", "bitmtp_linear_device_error",
        "bitmtp_linear_status_string", "bitmtp_linear_version", "bitmtp_linear_workspace_bytes",
        "bitmtp_linear_workspace_bytes_grouped", "bitmtp_linear_gemm_noalloc",
        "bitmtp_linear_ternarize_workspace_bytes", "bitmtp_linear_ternarize_pack",
        "bitmtp_linear_ternarize_workspace_bytes_grouped", "bitmtp_linear_ternarize_pack_grouped",
    }
    for s in syms:
        assert hasattr(lib, s), s
        assert hasattr(L, s), s  # binding keeps the C names


def test_binding_constants_match_header():
    """Every integer #define of the header has the same value in the binding."""
    import re
    text = open(L.HEADER_PATH).read()
    defs = {}
    for name, val in re.findall(r"^#define BITMTP_(\w+)\s+(\(?-?(?:0x)?[0-9a-fA-F]+u?\)?)", text, re.M):
        defs[name] = int(val.strip("()").rstrip("u"), 0)
    assert len(defs) >= 18
    for name, val in defs.items():
        assert getattr(L, name) == val, name
    assert L.NOALLOC_SCRATCH_BYTES == 4 * 1024 * 1024


def test_version_and_status_strings(lib):
    assert L.bitmtp_linear_version() == 0x000100
    for st in (L.OK, L.ERR_INVALID, L.ERR_ALIGN, L.ERR_SHAPE, L.ERR_NOT_TERNARY,
               L.ERR_UNSUPPORTED, L.ERR_CUDA, L.ERR_DEVICE, L.ERR_NOT_FINITE):
        assert L.status_string(st).startswith("BITMTP")
    assert "unknown" in L.status_string(12345)


@pytest.mark.parametrize("N,K", [(1, 1), (2560, 2560), (640, 2560), (32000, 2560), (4096, 11008),
                                 (129, 130), (7, 300)])
def test_packed_bytes_matches_oracle_definition(lib, N, K):
    assert L.packed_bytes(N, K) == oracle.packed_bytes(N, K)


def test_ternarize_validation(lib):
    """Argument checks of the device ternarisation, all before any CUDA call."""
    wb = L.bitmtp_linear_ternarize_workspace_bytes
    assert wb(0, 5) == 0 and wb(5, 0) == 0 and wb(5, L.MAX_K + 1) == 0
    assert wb(1, 1) == wb(700, 64) == wb(100000, L.MAX_K) == 512 * 8 + 256  # 512 bins + flag
    nb = L.packed_bytes(64, 64)
    tp = L.bitmtp_linear_ternarize_pack

    def call(W=FAKE, N=64, K=64, ldw=64, pk=FAKE, pk_bytes=nb, g=FAKE, ws=FAKE, ws_bytes=None):
        return tp(W, N, K, ldw, pk, pk_bytes, g, ws, wb(64, 64) if ws_bytes is None else ws_bytes, None)

    assert call(N=0) == L.ERR_SHAPE
    assert call(K=L.MAX_K + 1) == L.ERR_SHAPE
    assert call(W=None) == L.ERR_INVALID
    assert call(g=None) == L.ERR_INVALID
    assert call(ws=None) == L.ERR_INVALID
    assert call(ldw=63) == L.ERR_INVALID
    assert call(pk=FAKE + 8) == L.ERR_ALIGN
    assert call(ws=FAKE + 4) == L.ERR_ALIGN
    assert call(pk_bytes=nb - 1) == L.ERR_SHAPE
    assert call(ws_bytes=wb(64, 64) - 1) == L.ERR_SHAPE
    assert "NaN" in L.status_string(L.ERR_NOT_FINITE)


def test_ternarize_grouped_validation(lib):
    """Argument checks of the grouped ternarisation, all before any CUDA call."""
    wbg = L.bitmtp_linear_ternarize_workspace_bytes_grouped
    assert wbg(0) == 0 and wbg(L.MAX_GROUP + 1) == 0
    assert wbg(1) == L.bitmtp_linear_ternarize_workspace_bytes(64, 64)
    assert wbg(7) == 7 * 512 * 8 + 256
    nb = L.packed_bytes(64, 64)

    def call(n=2, ws=FAKE, ws_bytes=None, **kw):
        base = dict(W=FAKE, N=64, K=64, ldw=64, pk=FAKE, pk_bytes=nb, w_scale=FAKE)
        descs = [L.TernDesc(**base) for _ in range(n)]
        for k, v in kw.items():
            setattr(descs[-1], k, v)
        arr = (L.TernDesc * max(n, 1))(*descs) if n else None
        return L.bitmtp_linear_ternarize_pack_grouped(arr, n, ws, wbg(max(n, 1)) if ws_bytes is None else ws_bytes,
                                                      None)

    assert call(n=0) == L.ERR_INVALID
    assert call(n=L.MAX_GROUP + 1) == L.ERR_INVALID
    assert call(ws=None) == L.ERR_INVALID
    assert call(ws=FAKE + 4) == L.ERR_ALIGN
    assert call(ws_bytes=wbg(2) - 1) == L.ERR_SHAPE
    assert call(N=0) == L.ERR_SHAPE
    assert call(K=L.MAX_K + 1) == L.ERR_SHAPE
    assert call(W=None) == L.ERR_INVALID
    assert call(w_scale=None) == L.ERR_INVALID
    assert call(ldw=63) == L.ERR_INVALID
    assert call(pk=FAKE + 8) == L.ERR_ALIGN
    assert call(pk_bytes=nb - 1) == L.ERR_SHAPE


def test_packed_bytes_rejects(lib):
    assert L.packed_bytes(0, 5) == 0
    assert L.packed_bytes(5, 0) == 0
    assert L.packed_bytes(5, L.MAX_K + 1) == 0


def _act(kind=L.F32, x=FAKE, ldx=64, a_scale=None):
    return L.Act(kind, x, ldx, a_scale)


def _out(dtype=L.F32, y=FAKE, ldy=64, acc=None, lda=0):
    return L.Out(dtype, y, ldy, acc, lda)


WS = 1 << 24  # claimed workspace size for validation-only calls


def gemm(pk=FAKE, w=0.02, N=64, K=64, M=4, act=None, out=None, flags=0, ws=FAKE, ws_bytes=WS):
    act = act or _act()
    out = out or _out()
    return L.bitmtp_linear_gemm(pk, w, N, K, M, act, out, ws, ws_bytes, flags, None)


def test_gemm_validation(lib):
    assert gemm(M=17) == L.ERR_SHAPE
    assert gemm(M=-1) == L.ERR_SHAPE
    assert gemm(K=0) == L.ERR_SHAPE
    assert gemm(K=L.MAX_K + 1) == L.ERR_SHAPE
    assert gemm(N=-3) == L.ERR_SHAPE
    assert gemm(pk=None) == L.ERR_INVALID
    assert gemm(pk=FAKE + 8) == L.ERR_ALIGN
    assert gemm(act=_act(kind=7)) == L.ERR_INVALID
    assert gemm(act=_act(x=None)) == L.ERR_INVALID
    assert gemm(act=_act(ldx=63)) == L.ERR_INVALID
    assert gemm(act=_act(kind=L.Q8)) == L.ERR_INVALID          # Q8 without a_scale
    assert gemm(out=_out(dtype=5)) == L.ERR_INVALID
    assert gemm(out=_out(y=None)) == L.ERR_INVALID
    assert gemm(out=_out(ldy=10)) == L.ERR_INVALID
    assert gemm(out=_out(acc=FAKE, lda=3)) == L.ERR_INVALID
    assert gemm(w=float("nan")) == L.ERR_INVALID
    assert gemm(flags=L.FLAG_FORCE_TC | L.FLAG_FORCE_DP) == L.ERR_INVALID
    # FP8 activations: raw rows only, never the dp4a path
    assert gemm(act=_act(kind=L.Q8, a_scale=FAKE), flags=L.FLAG_FP8) == L.ERR_INVALID
    assert gemm(flags=L.FLAG_FP8 | L.FLAG_FORCE_DP) == L.ERR_INVALID
    assert gemm(M=0, act=_act(kind=L.Q8, a_scale=FAKE), flags=L.FLAG_FP8) == L.OK  # empty: a no-op
    assert gemm(M=17, flags=L.FLAG_FP8) == L.ERR_SHAPE
    assert L.load().bitmtp_linear_gemm(FAKE, 0.02, 64, 64, 4, None, ctypes.byref(_out()), FAKE, WS, 0,
                                       None) == L.ERR_INVALID
    assert gemm(ws=None) == L.ERR_INVALID
    assert gemm(ws=FAKE + 4) == L.ERR_ALIGN
    assert gemm(ws_bytes=L.bitmtp_linear_workspace_bytes(64, 64, 4) - 1) == L.ERR_SHAPE
    # empty problems are valid no-ops and never touch the device
    assert gemm(M=0) == L.OK
    assert gemm(N=0) == L.OK


def test_grouped_validation(lib):
    good = L.GemmDesc(FAKE, 0.02, 64, 64, 4, _act(), _out())
    bad = L.GemmDesc(FAKE, 0.02, 64, 64, 20, _act(), _out())
    grp = L.bitmtp_linear_gemm_grouped
    assert grp([good, bad], FAKE, WS, 0, None) == L.ERR_SHAPE
    assert grp([good] * (L.MAX_GROUP + 1), FAKE, WS, 0, None) == L.ERR_SHAPE
    assert grp([], FAKE, WS, 0, None) == L.OK
    empty = L.GemmDesc(FAKE, 0.02, 64, 64, 0, _act(), _out())
    assert grp([empty], None, 0, 0, None) == L.OK
    assert grp([good], None, 0, 0, None) == L.ERR_INVALID
    need = L.bitmtp_linear_workspace_bytes_grouped([good, good])
    assert grp([good, good], FAKE, need - 16, 0, None) == L.ERR_SHAPE
    q8 = L.GemmDesc(FAKE, 0.02, 64, 64, 4, _act(kind=L.Q8, a_scale=FAKE), _out())
    assert grp([good, q8], FAKE, WS, L.FLAG_FP8, None) == L.ERR_INVALID
    assert grp([good], FAKE, WS, L.FLAG_FP8 | L.FLAG_FORCE_DP, None) == L.ERR_INVALID


def test_workspace_bytes(lib):
    wb = L.bitmtp_linear_workspace_bytes
    assert wb(0, 64, 4) == 0 and wb(64, 0, 4) == 0 and wb(64, 64, 0) == 0 and wb(64, 64, 17) == 0
    a256 = lambda x: -(-x // 256) * 256
    # a 256-byte header, one ready flag (on its own 128-byte line) and one
    # partial-sum slot (16 rows x 128 columns of int32) per CTA of the largest
    # grid, then one activation region per problem: 4.5 KiB per k tile, prefix
    # sums of 16 rows, 16 scales
    fixed = 256 + 320 * 128 + 320 * 16 * 128 * 4
    region = lambda kt: a256(kt * 4608) + a256(16 * (kt + 1) * 4) + 256
    assert wb(128, 128, 1) == fixed + region(1)
    assert wb(32000, 2560, 16) == fixed + region(20)
    assert wb(32000, 2560, 1) == wb(5, 2560, 16)   # depends on K only
    d = [L.GemmDesc(FAKE, 0.02, 2560, 2560, 8, _act(ldx=2560), _out(ldy=2560)),
         L.GemmDesc(FAKE, 0.02, 640, 6912, 8, _act(ldx=6912), _out(ldy=640))]
    assert L.bitmtp_linear_workspace_bytes_grouped(d) == fixed + region(20) + region(54)
    bad = [L.GemmDesc(FAKE, 0.02, 2560, 2560, 20, _act(ldx=2560), _out(ldy=2560))]
    assert L.bitmtp_linear_workspace_bytes_grouped(bad) == 0


def test_noalloc_validation(lib):
    na = L.bitmtp_linear_gemm_noalloc
    assert na(FAKE, 0.02, 64, 64, 17, _act(), _out(), 0, None) == L.ERR_SHAPE
    assert na(FAKE, 0.02, 64, L.MAX_K + 1, 4, _act(), _out(), 0, None) == L.ERR_SHAPE
    assert na(FAKE, 0.02, 64, 64, 8, _act(), _out(), L.FLAG_FORCE_DP, None) == L.ERR_SHAPE
    assert na(FAKE, 0.02, 64, 64, 8, _act(kind=L.Q8, a_scale=FAKE), _out(), L.FLAG_FP8, None) == L.ERR_INVALID
    assert na(None, 0.02, 64, 64, 4, _act(), _out(), 0, None) == L.ERR_INVALID
    assert na(FAKE, 0.02, 64, 64, 0, _act(), _out(), 0, None) == L.OK
    # the built-in array covers the workspace of every shape inside the limits
    assert L.bitmtp_linear_workspace_bytes(L.MAX_N, L.MAX_K, L.MAX_M) <= L.NOALLOC_SCRATCH_BYTES
    assert "NOALLOC_SCRATCH_BYTES ((size_t)4 * 1024 * 1024)" in open(L.HEADER_PATH).read()


def test_pack_and_quant_validation(lib):
    pk = L.bitmtp_linear_pack
    assert pk(FAKE, 0, 16, 16, FAKE, 4096 + 16, None) == L.ERR_SHAPE
    assert pk(None, 4, 16, 16, FAKE, 4096 + 16, None) == L.ERR_INVALID
    assert pk(FAKE, 4, 16, 8, FAKE, 4096 + 16, None) == L.ERR_INVALID
    assert pk(FAKE, 4, 16, 16, FAKE + 4, 4096 + 16, None) == L.ERR_ALIGN
    assert pk(FAKE, 4, 16, 16, FAKE, 4096, None) == L.ERR_SHAPE   # trailer does not fit
    qa = L.bitmtp_linear_quant_act
    assert qa(FAKE, L.Q8, 2, 16, 16, FAKE, 16, FAKE, None, None) == L.ERR_INVALID
    assert qa(FAKE, L.F32, 2, 0, 16, FAKE, 16, FAKE, None, None) == L.ERR_SHAPE
    assert qa(FAKE, L.F32, 2, 16, 8, FAKE, 16, FAKE, None, None) == L.ERR_INVALID
    assert qa(FAKE, L.F32, 2, 16, 16, None, 16, FAKE, None, None) == L.ERR_INVALID
    assert qa(FAKE, L.F32, 0, 16, 16, None, 16, None, None, None) == L.OK


@pytest.mark.skipif(torch.cuda.is_available(), reason="checks the no-device answer")
def test_valid_calls_without_device_report_unsupported(lib):
    assert gemm() == L.ERR_UNSUPPORTED
    assert L.bitmtp_linear_gemm_noalloc(FAKE, 0.02, 64, 64, 4, _act(), _out(), 0, None) == L.ERR_UNSUPPORTED
    assert L.bitmtp_linear_quant_act(FAKE, L.F32, 2, 16, 16, FAKE, 16, FAKE, None, None) == L.ERR_UNSUPPORTED
    assert L.bitmtp_linear_pack(FAKE, 4, 16, 16, FAKE, 4096 + 16, None) == L.ERR_UNSUPPORTED
    assert L.bitmtp_linear_device_error(0) == L.ERR_UNSUPPORTED
