"""The C-ABI library loads, exports every entry point include/moe_ffn.h
declares, and rejects bad arguments on the host (no GPU needed: these checks
run before any CUDA call)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def M():
    import __graft_entry__
    __graft_entry__.build()
    import moe_expert_ffn_rms_gb300 as M
    return M


def _declared():
    names = []
    for fn in os.listdir(os.path.join(ROOT, "include")):
        if fn.endswith(".h"):
            src = open(os.path.join(ROOT, "include", fn)).read()
            src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
            names += re.findall(r"\b(moe_\w+)\s*\(", src)
    return sorted(set(names))


def test_every_declared_symbol_is_exported(M):
    declared = _declared()
    assert len(declared) >= 15
    for name in declared:
        assert hasattr(M.lib, name), name
    assert set(M.EXPORTED) >= set(declared)


def test_library_resolves_every_symbol_at_load(M):
    # RTLD_NOW binds every undefined symbol immediately: a missing definition
    # fails here instead of at the first call on a GPU machine.
    ctypes.CDLL(M.LIB_PATH, mode=os.RTLD_NOW)


def test_launch_counter_host_only(M):
    # host-side counter: readable without a GPU, and nothing launched here
    n = M.lib.moe_launch_count()
    assert n >= 0
    assert M.lib.moe_rmsnorm(None, None, 4, 256, 1e-6, None, None, None, None) == 1
    assert M.lib.moe_launch_count() == n  # a rejected call enqueues nothing


def test_abi_version_and_status_strings(M):
    assert M.abi_version() == 1
    assert M.lib.moe_status_string(0) == b"MOE_OK"
    assert M.lib.moe_status_string(6) == b"MOE_ERR_TIMEOUT"


def test_workspace_size_host_logic(M):
    ok = M.make_shape(16, 4096, 64, 1536, 8)
    n = M.moe_ffn_workspace_size(ok)
    # at least x_hat, x_p, the intermediate and the bf16 FC2 output rows
    R = 16 * 8
    assert n >= 16 * 4096 * 2 + R * 4096 * 2 + R * 1536 * 2 + R * 4096 * 2
    n8 = M.moe_ffn_workspace_size(M.make_shape(16, 4096, 64, 1536, 8, fp8=True))
    assert n8 > 0
    for bad in (M.make_shape(16, 100, 64, 1536, 8),   # H not a multiple of 64
                M.make_shape(16, 4096, 64, 1536, 9),  # top_k > 8
                M.make_shape(16, 4096, 4, 1536, 8),   # top_k > E
                M.make_shape(16, 4096, 300, 1536, 8)):  # E > 256
        assert M.lib.moe_ffn_workspace_size(ctypes.byref(bad)) == 0
        assert M.last_error()


def test_forward_rejects_bad_arguments_on_host(M):
    shape = M.make_shape(4, 256, 8, 512, 2)
    fake = 1 << 20  # 16-byte aligned non-null address; never dereferenced
    args = dict(x=fake, norm_w=fake, router_w=fake, router_logits=None, router_bias=None,
                w13=fake, w2=fake, w13_scale=None, w2_scale=None, out=fake, ids=None, tw=None,
                ws=fake, wsb=1 << 40)

    def call(**kw):
        a = dict(args, **kw)
        return M.lib.moe_ffn_forward(ctypes.byref(shape), a["x"], a["norm_w"], a["router_w"],
                                     a["router_logits"], a["router_bias"], a["w13"], a["w2"],
                                     a["w13_scale"], a["w2_scale"], a["out"], a["ids"], a["tw"],
                                     a["ws"], a["wsb"], None)
    assert call(x=None) == 1
    assert "non-NULL" in M.last_error()
    assert call(router_w=None) == 1            # neither router input
    assert call(router_logits=fake) == 1       # both router inputs
    assert call(x=fake + 8) == 1               # misaligned
    assert call(ws=fake + 16) == 1             # workspace not 256-aligned
    assert call(wsb=16) == 4                   # workspace too small
    bad = M.make_shape(4, 250, 8, 512, 2)
    assert M.lib.moe_ffn_forward(ctypes.byref(bad), fake, fake, fake, None, None, fake, fake, None,
                                 None, fake, None, None, fake, 1 << 40, None) == 2
    f8 = M.make_shape(4, 256, 8, 512, 2, fp8=True)
    assert M.lib.moe_ffn_forward(ctypes.byref(f8), fake, fake, fake, None, None, fake, fake, None,
                                 None, fake, None, None, fake, 1 << 40, None) == 1
    # FP8 weight scales must be 16-byte aligned (the tile epilogues read them as float4)
    assert M.lib.moe_ffn_forward(ctypes.byref(f8), fake, fake, fake, None, None, fake, fake,
                                 fake + 4, fake, fake, None, None, fake, 1 << 40, None) == 1
    assert "scales must be 16-byte aligned" in M.last_error()
    assert M.lib.moe_grouped_gemm(ctypes.byref(f8), 1, fake, fake, fake, fake + 8, fake, None, None,
                                  fake, None) == 1


def test_step_entry_points_reject_bad_arguments_on_host(M):
    fake = 1 << 20
    assert M.lib.moe_rmsnorm(None, fake, 4, 256, 1e-6, fake, None, None, None) == 1
    assert M.lib.moe_rmsnorm(fake, fake, 4, 250, 1e-6, fake, None, None, None) == 2
    assert M.lib.moe_rmsnorm(fake, fake, 4, 256, 1e-6, fake, fake, None, None) == 1
    assert M.lib.moe_route_topk(None, None, None, None, 4, 256, 8, 9, fake, fake, None, None, 0,
                                None) == 2
    assert M.lib.moe_route_topk(None, None, None, None, 4, 256, 8, 2, fake, fake, None, None, 0,
                                None) == 1
    assert M.lib.moe_permute(fake, 4, 300, 2, fake, fake, fake, None, None, 0, None, None, None, 0,
                             None) == 2
    assert M.lib.moe_permute(fake, 4, 8, 2, fake, fake, fake, fake, None, 0, None, None, None, 0,
                             None) == 1
    # a large batch needs the parallel sort's workspace
    assert M.lib.moe_permute_workspace_size(4096, 64, 8) == 128 * 64 * 4
    assert M.lib.moe_permute_workspace_size(16, 64, 8) == 0
    assert M.lib.moe_permute(fake, 4096, 64, 8, fake, fake, fake, None, None, 0, None, None, None,
                             0, None) == 4
    assert M.lib.moe_silu_and_mul(fake, 4, 12, fake, None) == 2
    assert M.lib.moe_combine(fake, 0, 0, fake, 4, 9, 256, fake, None) == 2
    assert M.lib.moe_combine(fake, 1, 1, fake, 4, 2, 252, fake, None) == 2
    assert M.lib.moe_quantize_fp8_rows(fake, 4, 20, fake, fake, None) == 2
    shape = M.make_shape(4, 256, 8, 512, 2)
    assert M.lib.moe_grouped_gemm(ctypes.byref(shape), 7, fake, None, fake, None, fake, None,
                                  None, fake, None) == 1
    assert M.lib.moe_grouped_ffn(ctypes.byref(shape), fake, None, fake, None, fake, None, fake,
                                 fake, fake, fake, fake, fake, 16, None) == 4
    assert M.lib.moe_grouped_ffn(ctypes.byref(shape), None, None, fake, None, fake, None, fake,
                                 fake, fake, fake, fake, fake, 1 << 20, None) == 1
    assert M.lib.moe_selftest_wait_timeout(0, None) == 1
    # NVFP4: H and I multiples of 256, only through the NVFP4 entry points
    nv_bad = M.make_shape(4, 320, 8, 256, 2, nvfp4=True)
    assert M.lib.moe_ffn_workspace_size(ctypes.byref(nv_bad)) == 0
    nv = M.make_shape(4, 256, 8, 256, 2, nvfp4=True)
    assert M.lib.moe_ffn_workspace_size(ctypes.byref(nv)) > 0
    assert M.lib.moe_ffn_forward(ctypes.byref(nv), fake, fake, fake, None, None, fake, fake, None,
                                 None, fake, None, None, fake, 1 << 40, None) == 1
    assert M.lib.moe_ffn_forward_nvfp4(ctypes.byref(shape), fake, fake, fake, None, None, fake, fake,
                                       fake, fake, fake, fake, fake, None, None, fake, 1 << 40,
                                       None) == 1          # shape not NVFP4
    assert M.lib.moe_ffn_forward_nvfp4(ctypes.byref(nv), fake, fake, fake, None, None, fake, None,
                                       fake, fake, fake, fake, fake, None, None, fake, 1 << 40,
                                       None) == 1          # block scales missing
    assert M.lib.moe_quantize_nvfp4(fake, 2, 4, 24, fake, fake, fake, None) == 2   # K % 16
    assert M.lib.moe_grouped_gemm(ctypes.byref(nv), 1, fake, None, fake, None, fake, None, None,
                                  fake, None) == 1
    # block-wise FP8: H % 256, I % 128, tiles of 1 or 128 rows by 128 columns
    fb_bad = M.make_shape(4, 384, 8, 256, 2, fp8="block")
    assert M.lib.moe_ffn_workspace_size(ctypes.byref(fb_bad)) == 0
    fb_bad_i = M.make_shape(4, 256, 8, 192, 2, fp8="block")
    assert M.lib.moe_ffn_workspace_size(ctypes.byref(fb_bad_i)) == 0
    fb = M.make_shape(4, 512, 8, 384, 2, fp8="block")
    assert fb.wdtype == M.W_FP8_BLOCK == 3
    n_fb = M.moe_ffn_workspace_size(fb)
    assert n_fb >= 4 * 512 * 2 + 4 * 512 + 4 * 4 * 4 + 8 * 512 + 8 * 4 * 4 + 8 * 384 + 8 * 3 * 4
    assert M.lib.moe_ffn_forward(ctypes.byref(fb), fake, fake, fake, None, None, fake, fake, None,
                                 None, fake, None, None, fake, 1 << 40, None) == 1  # scales missing
    assert M.lib.moe_grouped_gemm(ctypes.byref(fb), 1, fake, fake, fake, fake, fake, None, None,
                                  fake, None) == 1
    assert M.lib.moe_grouped_ffn_workspace_size(ctypes.byref(fb)) >= 8 * 3 * 4
    assert M.lib.moe_quantize_fp8_blocks(fake, 256, 200, 128, fake, fake, None) == 2  # K % 128
    assert M.lib.moe_quantize_fp8_blocks(fake, 200, 256, 128, fake, fake, None) == 2  # N % 128
    assert M.lib.moe_quantize_fp8_blocks(fake, 4, 256, 64, fake, fake, None) == 1   # block_rows
    assert M.lib.moe_quantize_fp8_blocks(None, 4, 256, 1, fake, fake, None) == 1
    assert M.lib.moe_route_workspace_size(4, 256, 8) > 0
    assert M.lib.moe_route_workspace_size(4, 250, 8) == 0


def test_no_gpu_reports_device_error(M):
    import torch
    if torch.cuda.is_available():
        pytest.skip("GPU present")
    rc = M.lib.moe_check_device()
    assert rc in (3, 5)
    assert M.last_error()
