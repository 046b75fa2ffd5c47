"""CPU-only checks of the C ABI: the library loads, exports every symbol the
header declares, and rejects bad arguments before touching a GPU."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "ra.h")


@pytest.fixture(scope="module")
def ra():
    import __graft_entry__
    __graft_entry__.build()
    import blockwise_exact_attention_ra_gb300 as ra
    return ra


def declared_symbols():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(ra_[a-z_0-9]+)\s*\(", text)))


def test_header_declares_the_entry_points():
    syms = declared_symbols()
    for need in ("ra_block_fwd", "ra_merge", "ra_ring_fwd", "ra_ring_bwd", "ra_finalize",
                 "ra_acc_init", "ra_sync_status", "ra_last_error"):
        assert need in syms


def test_library_exports_every_declared_symbol(ra):
    lib = ctypes.CDLL(ra._LIBPATH)
    for s in declared_symbols():
        assert hasattr(lib, s), s
        assert hasattr(ra, s), f"binding lacks {s}"


def test_workspace_sizes(ra):
    sh = ra.RaShape(1, 1024, 1024, 4, 2, 128, 0, 0)
    assert ra.ra_ring_fwd_workspace_bytes(ra.RA_BF16, sh, 4) >= 1024 * 2 * 128 * 2
    assert ra.ra_ring_fwd_workspace_bytes(ra.RA_F16, sh, 4) == 256   # the unit counter
    assert ra.ra_ring_fwd_workspace_bytes(ra.RA_F32, sh, 4) == 0
    ws = ra.ra_ring_bwd_workspace_bytes(ra.RA_BF16, ra.RA_F32, sh, 4)
    # D, LSE*log2e, fp32 dq accumulator, fp16 copies of q, k, v, dO
    need = 2 * 4 * 1024 * 4 + 1024 * 4 * 128 * 4 + 2 * (1024 * 4 * 128 * 2) + 2 * (1024 * 2 * 128 * 2)
    assert ws >= need
    assert ra.ra_ring_bwd_workspace_bytes(ra.RA_F32, ra.RA_F32, sh, 4) == 4 * 1024 * 4
    assert ra.ra_block_fwd_workspace_bytes(ra.RA_BF16, sh) >= 1024 * 2 * 128 * 2


def test_bad_shapes_are_rejected_without_a_gpu(ra):
    lib = ra.lib
    vp = ctypes.c_void_p(16)
    for sh in (ra.RaShape(0, 128, 128, 1, 1, 64, 0, 0),      # B = 0
               ra.RaShape(1, 128, 128, 3, 2, 64, 0, 0),      # Hq % Hkv != 0
               ra.RaShape(1, 128, 128, 2, 2, 0, 0, 0),       # d = 0
               ra.RaShape(1, 128, 128, 2, 2, 64, 5, 0)):     # batch stride < one batch
        rc = lib.ra_ring_fwd(vp, vp, vp, ra.RA_BF16, sh, 1, 1, 0.1, vp, ra.RA_F32, vp, None, 0, None)
        assert rc == 1, (sh.B, sh.Hq, sh.Hkv, sh.d)
        assert ra.ra_last_error()
    ok = ra.RaShape(1, 512, 512, 2, 2, 64, 0, 0)
    assert lib.ra_ring_fwd(vp, vp, vp, 7, ok, 1, 1, 0.1, vp, ra.RA_F32, vp, None, 0, None) == 1   # dtype
    assert lib.ra_ring_fwd(vp, vp, vp, ra.RA_BF16, ok, 3, 1, 0.1, vp, ra.RA_F32, vp, None, 0, None) == 1  # P
    assert lib.ra_ring_fwd(vp, vp, vp, ra.RA_BF16, ok, 1, 1, -1.0, vp, ra.RA_F32, vp, None, 0, None) == 1  # scale
    assert lib.ra_ring_fwd(vp, vp, vp, ra.RA_BF16, ok, 1, 1, float("nan"), vp, ra.RA_F32, vp, None, 0, None) == 1
    neq = ra.RaShape(1, 512, 256, 2, 2, 64, 0, 0)
    assert lib.ra_ring_fwd(vp, vp, vp, ra.RA_BF16, neq, 1, 1, 0.1, vp, ra.RA_F32, vp, None, 0, None) == 1
    odd = ra.RaShape(1, 384, 384, 2, 2, 64, 0, 0)   # host block 192 is not a multiple of 128
    assert lib.ra_ring_fwd(vp, vp, vp, ra.RA_BF16, odd, 2, 1, 0.1, vp, ra.RA_F32, vp, None, 0, None) == 2


def test_null_and_misaligned_pointers_are_rejected(ra):
    lib = ra.lib
    sh = ra.RaShape(1, 512, 512, 2, 2, 64, 0, 0)
    vp = ctypes.c_void_p(256)
    assert lib.ra_ring_fwd(None, vp, vp, ra.RA_BF16, sh, 1, 1, 0.1, vp, ra.RA_F32, vp, None, 0, None) == 1
    assert "q" in ra.ra_last_error()
    bad = ctypes.c_void_p(258)
    assert lib.ra_ring_fwd(vp, bad, vp, ra.RA_BF16, sh, 1, 1, 0.1, vp, ra.RA_F32, vp, None, 0, None) == 1
    assert "aligned" in ra.ra_last_error()
    assert lib.ra_merge(vp, vp, None, vp, vp, vp, sh, None) == 1
    assert lib.ra_block_fwd(vp, vp, vp, ra.RA_BF16, vp, vp, vp, sh, -1, 0, 1, 0.1, None, 0, None) == 1


def test_host_step_workspace_and_validation(ra):
    lib = ra.lib
    sh = ra.RaShape(2, 1024, 1024, 4, 2, 128, 0, 0)
    qel, kvel = 2 * 1024 * 4 * 128, 2 * 1024 * 2 * 128
    ws = ra.ra_ring_step_host_workspace_bytes(ra.RA_BF16, ra.RA_BF16, ra.RA_F32, sh, 4)
    # device copies (q, k, v, dO bf16; O bf16; LSE; dq, dk, dv fp32) + fwd and bwd workspaces
    copies = 2 * (2 * qel + 2 * kvel) + 2 * qel + 4 * 2 * 4 * 1024 + 4 * (qel + 2 * kvel)
    need = copies + ra.ra_ring_fwd_workspace_bytes(ra.RA_BF16, sh, 4) + \
        ra.ra_ring_bwd_workspace_bytes(ra.RA_BF16, ra.RA_F32, sh, 4)
    assert need <= ws <= need + 16 * 256
    assert ra.ra_ring_step_host_workspace_bytes(9, ra.RA_BF16, ra.RA_F32, sh, 4) == 0
    vp = ctypes.c_void_p(4096)
    wsz = ctypes.c_size_t(ws)

    def call(*, q=vp, flags=1, P=4, o=vp, workspace=vp, nbytes=wsz, shape=sh):
        return lib.ra_ring_step_host(q, vp, vp, vp, ra.RA_BF16, shape, P, flags, 0.1, o, ra.RA_BF16, vp,
                                     vp, vp, vp, ra.RA_F32, workspace, nbytes, None)
    assert call(flags=8) == 1 and "flag" in ra.ra_last_error()
    assert call(P=3) == 1
    assert call(q=None) == 1 and "q" in ra.ra_last_error()
    assert call(o=None) == 1
    assert call(nbytes=ctypes.c_size_t(ws - 1)) == 1 and "workspace" in ra.ra_last_error()
    assert call(workspace=ctypes.c_void_p(4096 + 16)) == 1 and "aligned" in ra.ra_last_error()
    assert call(shape=ra.RaShape(2, 1024, 1024, 3, 2, 128, 0, 0)) == 1


def test_ffn_validation(ra):
    lib = ra.lib
    vp = ctypes.c_void_p(4096)
    ws = ra.ra_ffn_workspace_bytes(ra.RA_BF16, 1024, 512, 2048, 256, True)
    assert ws >= 3 * 256 * 2048 * 2
    assert ra.ra_ffn_workspace_bytes(ra.RA_BF16, 1024, 512, 2048, 256, False) >= 256 * 2048 * 2
    assert ra.ra_ffn_workspace_bytes(ra.RA_F32, 1024, 512, 2048, 256, False) == 0   # fp32 not taken
    wsz = ctypes.c_size_t(ws)

    def fwd(*, dtype=ra.RA_BF16, T=1024, dm=512, dh=2048, block=256, x=vp, nbytes=wsz):
        return lib.ra_ffn_fwd(x, vp, vp, dtype, T, dm, dh, block, vp, ra.RA_F32, vp, nbytes, None)
    assert fwd(dtype=ra.RA_F32) == 2
    assert fwd(dm=500) == 2 and fwd(dh=2000) == 2 and fwd(T=1000) == 2 and fwd(block=200) == 2
    assert fwd(T=0) == 1
    assert fwd(x=None) == 1 and "x" in ra.ra_last_error()
    assert fwd(nbytes=ctypes.c_size_t(16)) == 1 and "workspace" in ra.ra_last_error()
    assert lib.ra_ffn_bwd(vp, vp, vp, None, ra.RA_BF16, 1024, 512, 2048, 256, vp, ra.RA_F32, vp, vp, vp,
                          wsz, None) != 0


def test_rejected_flag_combinations(ra):
    lib = ra.lib
    sh = ra.RaShape(1, 1024, 1024, 2, 2, 128, 0, 0)
    vp = ctypes.c_void_p(4096)
    hl = ctypes.c_void_p(8192)
    both = ra.RA_CAUSAL | ra.RA_STRIPED
    # the striped layout and per-host lengths do not combine
    assert lib.ra_ring_fwd_varlen(vp, vp, vp, ra.RA_BF16, sh, 4, hl, both, 0.1, vp, ra.RA_F32, vp, vp,
                                  ctypes.c_size_t(1 << 30), None) == 1
    assert "STRIPED" in ra.ra_last_error()
    assert lib.ra_ring_bwd_varlen(vp, vp, vp, vp, ra.RA_F32, vp, vp, ra.RA_BF16, sh, 4, hl, both, 0.1, vp, vp, vp,
                                  ra.RA_F32, vp, ctypes.c_size_t(1 << 30), None) == 1
    # a missing or misaligned length array
    assert lib.ra_ring_fwd_varlen(vp, vp, vp, ra.RA_BF16, sh, 4, None, 1, 0.1, vp, ra.RA_F32, vp, vp,
                                  ctypes.c_size_t(1 << 30), None) == 1
    assert lib.ra_ring_fwd_varlen(vp, vp, vp, ra.RA_BF16, sh, 4, ctypes.c_void_p(8194), 1, 0.1, vp, ra.RA_F32,
                                  vp, vp, ctypes.c_size_t(1 << 30), None) == 1
    # unknown flag bits
    assert lib.ra_ring_fwd(vp, vp, vp, ra.RA_BF16, sh, 4, 64, 0.1, vp, ra.RA_F32, vp, vp, ctypes.c_size_t(1 << 30),
                           None) == 1


def test_launch_counter_is_readable(ra):
    assert isinstance(ra.ra_launch_count(), int) and ra.ra_launch_count() >= 0


def test_visit_log_arguments_are_checked(ra):
    lib = ra.lib
    # turning the log off always succeeds; a log without a count word or with a
    # misaligned entry array is refused before anything is recorded
    assert lib.ra_debug_visit_log(None, 0, None) == 0
    assert lib.ra_debug_visit_log(ctypes.c_void_p(4096), 16, None) == 1
    assert lib.ra_debug_visit_log(ctypes.c_void_p(4096), 0, ctypes.c_void_p(8192)) == 1
    assert lib.ra_debug_visit_log(ctypes.c_void_p(4104), 16, ctypes.c_void_p(8192)) == 1
    assert "aligned" in ra.ra_last_error()
    assert lib.ra_debug_visit_log(None, 0, None) == 0


def test_strides_are_checked_without_a_gpu(ra):
    lib = ra.lib
    vp = ctypes.c_void_p(16)
    assert len(ra.RaShape._fields_) == 12   # the header's ra_shape
    bad = (
        ra.RaShape(1, 256, 256, 2, 2, 64, 0, 0, 64, 64, 0, 0),      # rows and heads at the same stride
        ra.RaShape(1, 256, 256, 2, 2, 64, 0, 0, 32, 0, 0, 0),       # row stride shorter than a row
        ra.RaShape(1, 256, 256, 2, 2, 64, 0, 0, 64, 100, 0, 0),     # heads overlap the row block
        ra.RaShape(1, 256, 256, 2, 2, 64, 0, 0, -64, 0, 0, 0),      # negative stride
        ra.RaShape(2, 256, 256, 2, 2, 64, 1000, 0, 0, 0, 0, 0),     # batch shorter than its extent
        ra.RaShape(1, 256, 256, 2, 2, 64, 0, 0, 0, 0, 0, 32),       # kv heads overlap
    )
    for sh in bad:
        rc = lib.ra_ring_fwd(vp, vp, vp, ra.RA_BF16, sh, 1, 1, 0.1, vp, ra.RA_F32, vp, None, 0, None)
        assert rc == 1, (sh.q_rstride, sh.q_hstride, sh.kv_hstride)
        assert "stride" in ra.ra_last_error()
    # the host-buffer step takes packed rows only; [B, H, N, d] host tensors are refused
    hm = ra.RaShape(1, 256, 256, 2, 2, 64, 0, 0, 64, 256 * 64, 64, 256 * 64)
    ws = ctypes.c_void_p(1 << 20)
    rc = lib.ra_ring_step_host(vp, vp, vp, vp, ra.RA_BF16, hm, 2, 1, 0.1, vp, ra.RA_F32, vp, vp, vp, vp,
                               ra.RA_F32, ws, 1 << 40, None)
    assert rc == 2 and "packed rows" in ra.ra_last_error()


def test_binding_passes_tensor_strides(ra):
    import torch
    x = torch.zeros(2, 4, 96, 64)                         # [B, H, N, d]
    q = x.permute(0, 2, 1, 3)                             # viewed as [B, N, H, d]
    sh = ra.shape_of(q, q)
    assert (sh.q_bstride, sh.q_rstride, sh.q_hstride) == (4 * 96 * 64, 64, 96 * 64)
    one = torch.zeros(1, 96, 1, 64)
    sh1 = ra.shape_of(one, one)
    assert (sh1.q_bstride, sh1.q_hstride) == (0, 0)      # extent-1 axes take the default
    with pytest.raises(ra.RAError):
        ra._same_layout(torch.zeros(2, 96, 4, 64), q, "o", "q")
    assert ra.empty_like_layout(q).stride() == q.stride()
