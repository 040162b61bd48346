"""CPU checks of the C ABI: the library builds for sm_103a, loads, exports every
function the header declares, and rejects bad arguments before touching a GPU."""
import ctypes
import os
import re

import pytest

import causal_gqa_flash_gb300 as gqa

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "gqa_attn.h")


def declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return set(re.findall(r"\b(attn_[a-z0-9_]+)\s*\(", src))


@pytest.fixture(scope="module")
def lib():
    gqa.build()
    return gqa.load()


def test_header_matches_binding():
    assert declared_functions() == set(gqa.EXPORTED_SYMBOLS)


def test_library_exports_every_declared_symbol(lib):
    raw = ctypes.CDLL(gqa.library_path())
    for name in declared_functions():
        assert hasattr(raw, name), name


def test_version_and_workspace(lib):
    assert gqa.attn_version() == "0.1.0"
    # two fp32 arrays [B, Hq, T rounded up to 128] and 256 bytes of task counters
    assert gqa.attn_bwd_workspace_bytes(2, 3000, 6) == 2 * 2 * 6 * 3072 * 4 + 256  # two fp32 arrays + task counters
    assert gqa.attn_bwd_workspace_bytes(1, 128, 1) == 2 * 128 * 4 + 256
    assert gqa.attn_bwd_workspace_bytes(0, 128, 1) == 0


FAKE = ctypes.c_void_p(0x100000)      # aligned, never dereferenced: validation fails first
MISALIGNED = ctypes.c_void_p(0x100008)


@pytest.mark.parametrize("B,T,Hq,Hkv,d,needle", [
    (1, 128, 6, 2, 96, "d must be 64 or 128"),
    (1, 128, 5, 2, 64, "multiple of Hkv"),
    (1, 0, 6, 2, 64, "positive"),
    (0, 128, 6, 2, 64, "positive"),
    (1, 128, 6, 0, 64, "positive"),
])
def test_fwd_rejects_bad_shapes(lib, B, T, Hq, Hkv, d, needle):
    rc = lib.attn_fwd(FAKE, FAKE, FAKE, FAKE, FAKE, B, T, Hq, Hkv, d, 1, None)
    assert rc == gqa.GQA_ERR_INVALID_ARG
    assert needle in gqa.attn_last_error()


def test_fwd_rejects_null_and_misaligned(lib):
    rc = lib.attn_fwd(None, FAKE, FAKE, FAKE, FAKE, 1, 128, 6, 2, 64, 1, None)
    assert rc == gqa.GQA_ERR_INVALID_ARG and "q is NULL" in gqa.attn_last_error()
    rc = lib.attn_fwd(FAKE, FAKE, MISALIGNED, FAKE, FAKE, 1, 128, 6, 2, 64, 1, None)
    assert rc == gqa.GQA_ERR_INVALID_ARG and "v is not 16-byte aligned" in gqa.attn_last_error()


def test_bwd_rejects_small_workspace(lib):
    need = gqa.attn_bwd_workspace_bytes(2, 256, 4)
    args = [FAKE] * 10 + [need - 1, 2, 256, 4, 2, 64, 1, None]
    rc = lib.attn_bwd(*args)
    assert rc == gqa.GQA_ERR_INVALID_ARG and "workspace_bytes" in gqa.attn_last_error()
    args = [FAKE] * 9 + [None, need, 2, 256, 4, 2, 64, 1, None]
    rc = lib.attn_bwd(*args)
    assert rc == gqa.GQA_ERR_INVALID_ARG and "workspace is NULL" in gqa.attn_last_error()


def test_last_error_is_cleared_by_next_call(lib):
    lib.attn_fwd(None, None, None, None, None, 1, 128, 6, 2, 64, 1, None)
    assert gqa.attn_last_error()
    lib.attn_fwd(FAKE, FAKE, FAKE, FAKE, FAKE, 1, 128, 6, 2, 96, 1, None)
    assert "d must be" in gqa.attn_last_error()


def _view(ptr=FAKE, st=6 * 64, sb=128 * 6 * 64):
    return gqa.GqaView(ptr.value if isinstance(ptr, ctypes.c_void_p) else ptr, st, sb)


@pytest.mark.parametrize("st,sb,needle", [
    (6 * 64 + 4, 128 * 6 * 64, "multiples of 8"),   # token stride not 16-byte aligned
    (0, 128 * 6 * 64, "positive"),                  # zero token stride
    (-384, 128 * 6 * 64, "positive"),               # negative token stride
    (6 * 64, 1 << 39, "below 2^39"),                # batch stride out of TMA range
])
def test_strided_fwd_rejects_bad_strides(lib, st, sb, needle):
    rc = lib.attn_fwd_strided(_view(st=st, sb=sb), _view(st=2 * 64, sb=128 * 2 * 64), _view(st=2 * 64, sb=128 * 2 * 64),
                              _view(), FAKE, 2, 128, 6, 2, 64, 1, None)
    assert rc == gqa.GQA_ERR_INVALID_ARG
    assert needle in gqa.attn_last_error() and "q strides" in gqa.attn_last_error()


def test_strided_rejects_self_overlapping_output(lib):
    k = _view(st=2 * 64, sb=128 * 2 * 64)
    # token stride smaller than the H*d elements of one token: rows of o overlap
    rc = lib.attn_fwd_strided(_view(), k, k, _view(st=4 * 64, sb=128 * 6 * 64), FAKE, 2, 128, 6, 2, 64, 1, None)
    assert rc == gqa.GQA_ERR_INVALID_ARG and "output o overlaps itself" in gqa.attn_last_error()
    # batch stride smaller than one sequence while tokens are not interleaved with batches
    rc = lib.attn_fwd_strided(_view(), k, k, _view(st=6 * 64, sb=127 * 6 * 64), FAKE, 2, 128, 6, 2, 64, 1, None)
    assert rc == gqa.GQA_ERR_INVALID_ARG and "overlaps itself" in gqa.attn_last_error()
    # the same strides are fine for an input (never written)
    ok_in = _view(st=6 * 64, sb=127 * 6 * 64)
    rc = lib.attn_fwd_strided(ok_in, k, k, _view(st=4 * 64, sb=128 * 6 * 64), FAKE, 2, 128, 6, 2, 64, 1, None)
    assert "output o overlaps itself" in gqa.attn_last_error()


def test_strided_unused_strides_are_ignored(lib):
    """With B == 1 and T == 1 the batch and token strides are never used: any value passes
    validation, which then fails on the next check (a misaligned lse), not on the strides."""
    junk = _view(st=3, sb=-5)
    rc = lib.attn_fwd_strided(junk, junk, junk, junk, MISALIGNED, 1, 1, 6, 2, 64, 1, None)
    assert rc == gqa.GQA_ERR_INVALID_ARG and "lse is not 16-byte aligned" in gqa.attn_last_error()


def test_strided_bwd_checks_every_view(lib):
    need = gqa.attn_bwd_workspace_bytes(2, 128, 6)
    q, k = _view(), _view(st=2 * 64, sb=128 * 2 * 64)
    bad = _view(MISALIGNED)
    rc = lib.attn_bwd_strided(q, k, k, q, FAKE, q, q, k, bad, FAKE, need, 2, 128, 6, 2, 64, 1, None)
    assert rc == gqa.GQA_ERR_INVALID_ARG and "dv is not 16-byte aligned" in gqa.attn_last_error()
    rc = lib.attn_bwd_strided(q, k, k, q, FAKE, q, q, _view(st=2 * 64, sb=64), k, FAKE, need, 2, 128, 6, 2, 64, 1,
                              None)
    assert rc == gqa.GQA_ERR_INVALID_ARG and "output dk overlaps itself" in gqa.attn_last_error()
    rc = lib.attn_bwd_strided(q, k, k, q, FAKE, q, q, k, k, FAKE, need - 1, 2, 128, 6, 2, 64, 1, None)
    assert rc == gqa.GQA_ERR_INVALID_ARG and "workspace_bytes" in gqa.attn_last_error()


def test_rope_table_bytes_and_checks(lib):
    assert gqa.load().attn_rope_table_bytes(8192, 128) == 8192 * 64 * 2 * 4
    assert gqa.load().attn_rope_table_bytes(0, 64) == 0 and gqa.load().attn_rope_table_bytes(16, 96) == 0
    for T, d, base, ptr, needle in ((16, 96, 1e4, FAKE, "d must be 64 or 128"), (0, 64, 1e4, FAKE, "T must be"),
                                    (16, 64, 0.0, FAKE, "base must be positive"),
                                    (16, 64, float("nan"), FAKE, "base must be positive"),
                                    (16, 64, 1e4, None, "table is NULL"),
                                    (16, 64, 1e4, MISALIGNED, "table is not 16-byte aligned")):
        rc = lib.attn_rope_table(ptr, T, d, base, None)
        assert rc == gqa.GQA_ERR_INVALID_ARG and needle in gqa.attn_last_error(), needle


def test_rope_argument_checks(lib):
    x = _view(st=6 * 64, sb=128 * 6 * 64)
    rc = lib.attn_rope(x, x, FAKE, 2, 128, 6, 96, 0, None)
    assert rc == gqa.GQA_ERR_INVALID_ARG and "d must be 64 or 128" in gqa.attn_last_error()
    rc = lib.attn_rope(x, x, None, 2, 128, 6, 64, 0, None)
    assert rc == gqa.GQA_ERR_INVALID_ARG and "table is NULL" in gqa.attn_last_error()
    rc = lib.attn_rope(x, _view(st=6 * 64 + 8, sb=128 * 7 * 64), FAKE, 2, 128, 6, 64, 0, None)
    assert rc == gqa.GQA_ERR_INVALID_ARG and "same strides" in gqa.attn_last_error()
    rc = lib.attn_rope(x, _view(st=5 * 64, sb=128 * 6 * 64, ptr=0x200000), FAKE, 2, 128, 6, 64, 0, None)
    assert rc == gqa.GQA_ERR_INVALID_ARG and "output y overlaps itself" in gqa.attn_last_error()
    rc = lib.attn_rope(x, x, FAKE, 0, 128, 6, 64, 0, None)
    assert rc == gqa.GQA_ERR_INVALID_ARG and "positive" in gqa.attn_last_error()


def test_binding_checks_shapes_types_and_device_before_calling(lib):
    """The C ABI takes raw pointers and cannot see sizes: the binding refuses mismatched
    shapes, dtypes and non-CUDA tensors before any pointer reaches the library."""
    import torch
    bf = torch.bfloat16
    q, k = torch.zeros((1, 128, 6, 64), dtype=bf), torch.zeros((1, 128, 2, 64), dtype=bf)
    with pytest.raises(ValueError, match="does not match q"):
        gqa.attn_fwd(q, torch.zeros((1, 127, 2, 64), dtype=bf), k)
    with pytest.raises(ValueError, match="must have the shape of k"):
        gqa.attn_fwd(q, k, torch.zeros((1, 128, 3, 64), dtype=bf))
    with pytest.raises(ValueError, match="q must be torch.bfloat16"):
        gqa.attn_fwd(q.float(), k, k)
    with pytest.raises(ValueError, match="q must be contiguous"):
        gqa.attn_fwd(q.transpose(1, 2).contiguous().transpose(1, 2), k, k)
    with pytest.raises(ValueError, match="current CUDA device"):
        gqa.attn_fwd(q, k, k)
    with pytest.raises(ValueError, match="dO must have shape"):
        gqa.attn_bwd_dq(q, k, k, torch.zeros((1, 128, 5, 64), dtype=bf), q, None)


def test_naive_workspace_and_checks(lib):
    assert gqa.attn_naive_workspace_bytes(2, 100, 3) == 2 * 3 * 100 * 100 * (4 + 2 + 2)
    need = gqa.attn_naive_workspace_bytes(1, 128, 6)
    rc = lib.attn_fwd_naive(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, need - 1, 1, 128, 6, 2, 64, 1, None)
    assert rc == gqa.GQA_ERR_INVALID_ARG and "workspace_bytes" in gqa.attn_last_error()
    rc = lib.attn_bwd_naive(*([FAKE] * 10), need, 1, 128, 6, 2, 96, 1, None)
    assert rc == gqa.GQA_ERR_INVALID_ARG and "d must be 64 or 128" in gqa.attn_last_error()


def test_build_compiles_every_cuda_source():
    """build() compiles the library from an explicit list; a .cu file left out of it
    would silently drop its kernels (and C entry points) from the GPU machine's build."""
    from causal_gqa_flash_gb300 import _build
    on_disk = {f for f in os.listdir(_build.CSRC) if f.endswith(".cu")}
    assert on_disk == set(_build.SOURCES)


def test_kernel_source_hash_ignores_comments_only(tmp_path, monkeypatch):
    """The recorded DRAM traffic stays valid across comment edits and lapses on code edits."""
    import bench
    src = tmp_path / "causal_gqa_flash_gb300" / "csrc"
    src.mkdir(parents=True)
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    (src / "k.cu").write_text("int f() { return 1; }  // one\n/* block */\n")
    h0 = bench.kernel_source_hash(["k.cu"])
    (src / "k.cu").write_text("// a new comment\nint f() { return 1; }  // changed\n\n")
    assert bench.kernel_source_hash(["k.cu"]) == h0
    (src / "k.cu").write_text("int f() { return 2; }\n")
    assert bench.kernel_source_hash(["k.cu"]) != h0


def test_binding_checks_views_rope_and_naive_arguments(lib):
    """Shape and dtype mistakes in the strided, rotary and naive entry points are
    refused by the binding, before any pointer reaches the library."""
    import torch
    bf = torch.bfloat16
    q, k = torch.zeros((2, 64, 6, 64), dtype=bf), torch.zeros((2, 64, 2, 64), dtype=bf)
    lse = torch.zeros((2, 6, 64))
    with pytest.raises(ValueError, match="o must have shape"):
        gqa.attn_fwd_strided(q, k, k, torch.zeros((2, 64, 5, 64), dtype=bf))
    with pytest.raises(ValueError, match="dk must have shape"):
        gqa.attn_bwd_strided(q, k, k, q, lse, q, q, torch.zeros((2, 64, 3, 64), dtype=bf), k)
    with pytest.raises(ValueError, match="lse must have shape"):
        gqa.attn_bwd_strided(q, k, k, q, torch.zeros((2, 6, 63)), q, q, k, k)
    with pytest.raises(ValueError, match="does not cover"):
        gqa.attn_rope(q, torch.zeros((63, 32, 2)))          # table shorter than T
    with pytest.raises(ValueError, match="does not cover"):
        gqa.attn_rope(q, torch.zeros((64, 64, 2)))          # table for d = 128
    with pytest.raises(ValueError, match="y must have shape"):
        gqa.attn_rope(q, torch.zeros((64, 32, 2)), y=k)
    with pytest.raises(ValueError, match="table must be torch.float32"):
        gqa.attn_rope(q, torch.zeros((64, 32, 2), dtype=torch.float64))
    with pytest.raises(ValueError, match="must have the shape of k"):
        gqa.attn_fwd_naive(q, k, q)
    with pytest.raises(ValueError, match="lse must have shape"):
        gqa.attn_bwd_naive(q, k, k, q, torch.zeros((2, 6, 65)), q)


def test_fused_rope_argument_checks(lib):
    """attn_fwd_rope / attn_bwd_rope refuse bad views, a bad base and an in-place
    rotation whose strides differ, before any launch."""
    q, k = _view(), _view(st=2 * 64, sb=128 * 2 * 64)
    for base in (0.0, -1.0, float("nan"), float("inf")):
        rc = lib.attn_fwd_rope(q, k, k, q, FAKE, q, k, base, 2, 128, 6, 2, 64, 1, None)
        assert rc == gqa.GQA_ERR_INVALID_ARG and "base must be positive" in gqa.attn_last_error()
    rc = lib.attn_fwd_rope(q, k, k, q, FAKE, _view(st=6 * 64 + 64, sb=128 * 7 * 64), k, 1e4, 2, 128, 6, 2, 64, 1,
                           None)
    assert rc == gqa.GQA_ERR_INVALID_ARG and "q_rot == q" in gqa.attn_last_error()
    rc = lib.attn_fwd_rope(q, k, k, q, FAKE, _view(ptr=0x400000), _view(st=3 * 64, sb=128 * 3 * 64), 1e4, 2, 128,
                           6, 2, 64, 1, None)
    assert rc == gqa.GQA_ERR_INVALID_ARG and "k_rot == k" in gqa.attn_last_error()
    rc = lib.attn_fwd_rope(q, k, k, q, FAKE, _view(MISALIGNED), k, 1e4, 2, 128, 6, 2, 64, 1, None)
    assert rc == gqa.GQA_ERR_INVALID_ARG and "q_rot is not 16-byte aligned" in gqa.attn_last_error()
    rc = lib.attn_fwd_rope(q, k, k, q, FAKE, q, k, 1e4, 2, 128, 6, 4, 64, 1, None)
    assert rc == gqa.GQA_ERR_INVALID_ARG and "multiple" in gqa.attn_last_error()
    need = gqa.attn_bwd_workspace_bytes(2, 128, 6)
    rc = lib.attn_bwd_rope(q, k, k, q, FAKE, q, q, k, k, 0.0, FAKE, need, 2, 128, 6, 2, 64, 1, None)
    assert rc == gqa.GQA_ERR_INVALID_ARG and "base must be positive" in gqa.attn_last_error()
    rc = lib.attn_bwd_rope(q, k, k, q, FAKE, q, q, _view(st=2 * 64, sb=64), k, 1e4, FAKE, need, 2, 128, 6, 2, 64, 1,
                           None)
    assert rc == gqa.GQA_ERR_INVALID_ARG and "output dk overlaps itself" in gqa.attn_last_error()
    rc = lib.attn_bwd_rope(q, k, k, q, FAKE, q, q, k, k, 1e4, FAKE, need - 1, 2, 128, 6, 2, 64, 1, None)
    assert rc == gqa.GQA_ERR_INVALID_ARG and "workspace_bytes" in gqa.attn_last_error()


def test_binding_checks_fused_rope_arguments(lib):
    import torch
    bf = torch.bfloat16
    q, k = torch.zeros((2, 64, 6, 64), dtype=bf), torch.zeros((2, 64, 2, 64), dtype=bf)
    lse = torch.zeros((2, 6, 64))
    with pytest.raises(ValueError, match="k_rot must have shape"):
        gqa.attn_fwd_rope(q, k, k, k_rot=q)
    with pytest.raises(ValueError, match="q_rot must have shape"):
        gqa.attn_fwd_rope(q, k, k, q_rot=k)
    with pytest.raises(ValueError, match="lse must have shape"):
        gqa.attn_bwd_rope(q, k, k, q, torch.zeros((2, 6, 63)), q)
    with pytest.raises(ValueError, match="dk must have shape"):
        gqa.attn_bwd_rope(q, k, k, q, lse, q, dk=q)


def test_task_order_argument_checks(lib):
    assert lib.attn_set_task_order(3) == gqa.GQA_ERR_INVALID_ARG
    assert "order must be 0" in gqa.attn_last_error()
    assert lib.attn_set_task_order(-1) == gqa.GQA_ERR_INVALID_ARG
    for order in (1, 2, 0):
        assert lib.attn_set_task_order(order) == gqa.GQA_OK


def test_probe_tma_argument_checks(lib):
    buf = ctypes.c_void_p(0x10000)  # never dereferenced: every call below is refused first
    out = ctypes.c_void_p(0x20000)
    cases = [
        ((buf, 16384 + 128, 4, 1, 10, out), "multiple of 16384"),
        ((buf, 0, 4, 1, 10, out), "multiple of 16384"),
        ((buf, 1 << 20, 4, 3, 10, out), "ctas_per_sm must be 1 or 2"),
        ((buf, 1 << 20, 0, 1, 10, out), "stages must be in [1, 8]"),
        ((buf, 1 << 20, 9, 1, 10, out), "stages must be in [1, 8]"),
        ((buf, 1 << 20, 7, 2, 10, out), "stages must be in [1, 6]"),
        ((buf, 1 << 20, 4, 1, 0, out), "iters must be in"),
        ((None, 1 << 20, 4, 1, 10, out), "buf is NULL"),
        ((ctypes.c_void_p(0x10008), 1 << 20, 4, 1, 10, out), "not 16-byte aligned"),
    ]
    for args, needle in cases:
        assert lib.attn_probe_tma(*args, None) == gqa.GQA_ERR_INVALID_ARG, needle
        assert needle in gqa.attn_last_error(), (needle, gqa.attn_last_error())
