"""The C-ABI library on the host (no GPU): it loads, exports every declared symbol, and rejects
bad arguments with the documented status before anything touches a device."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "moe.h")


@pytest.fixture(scope="module")
def moe():
    from mixture_experts_sparse_02_b300 import build
    build.build()
    from mixture_experts_sparse_02_b300 import moe as m
    return m


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(moe_[a-z_]+)\s*\(", text)))


def test_exports_every_declared_symbol(moe):
    names = declared_functions()
    assert len(names) >= 11
    from mixture_experts_sparse_02_b300 import build
    for path in (moe.LIB_PATH, build.build(debug_bounds=True)):   # the normal and the bounds-checking build
        lib = ctypes.CDLL(path)
        for n in names:
            assert hasattr(lib, n), (path, n)
    assert set(names) == set(moe.EXPORTS)


C_CALLER = r"""
#include <stdio.h>
#include "moe.h"
/* A C99 caller: configure a Mixtral-shaped layer, size its workspace, and reference every
   declared entry point through a function pointer (nothing is called on a device). */
int main(void) {
  moe_config c = {4096, 4096, 14336, 8, 2, MOE_BF16, MOE_SOFTMAX_TOPK_RENORM, 0, 0, 0.0f};
  size_t ws = moe_workspace_bytes(&c);
  moe_status (*fwd)(const moe_config*, const void*, const void*, const float*, const float*, const void*,
                    const void*, const void*, const void*, const void*, const void*, void*, int32_t*, int32_t*,
                    void*, size_t, moe_stream_t) = moe_forward;
  printf("%zu %s %d %p\n", ws, moe_status_string(MOE_OK), MOE_NUM_STAGES, (void*)fwd);
  return ws > 0 ? 0 : 1;
}
"""


def test_header_compiles_and_links_as_c(moe, tmp_path):
    """include/moe.h is plain C: a C99 program includes it, type-checks a call signature and
    links against the library (it is not run: the library needs the CUDA driver)."""
    import shutil
    import subprocess
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    src = tmp_path / "caller.c"
    src.write_text(C_CALLER)
    lib_dir = os.path.dirname(moe.LIB_PATH)
    r = subprocess.run([cc, "-std=c99", "-Wall", "-Werror", "-I", os.path.join(ROOT, "include"), str(src),
                        "-o", str(tmp_path / "caller"), "-L", lib_dir, "-l:libmoe.so", "-Wl,--allow-shlib-undefined"],
                       capture_output=True, text=True)
    assert r.returncode == 0, r.stderr


def test_status_strings(moe):
    for s in range(6):
        assert moe.status_string(s) and moe.status_string(s) != "unknown status"


def test_workspace_bytes(moe):
    c = moe.config(4096, 4096, 14336, 8, 2)
    big = moe.workspace_bytes(c)
    assert big > 4096 * 2 * 4096 * 2  # at least x_perm
    assert moe.workspace_bytes(moe.config(64, 4096, 14336, 8, 2)) < big
    assert moe.workspace_bytes(moe.config(4, 64, 64, 8, 9)) == 0        # k > E: invalid
    s = moe.workspace_bytes(moe.config(8192, 7168, 2048, 256, 8, scoring="sigmoid", n_shared=1, d_ff_shared=2048))
    assert s > 8192 * 8 * 7168 * (2 + 4)            # x_perm (bf16) and y_perm (float32)


FAKE = 0x100000  # a 16-byte aligned address that is never dereferenced: the checks return first


def _gpu_visible() -> bool:
    try:
        import torch
        return torch.cuda.is_available()
    except Exception:
        return False


# The tests below pass FAKE for device pointers and expect the host-side checks to refuse the
# call before any launch.  They run only where no GPU is visible, so that a regressed check
# cannot launch a kernel on a fabricated address.
host_only = pytest.mark.skipif(_gpu_visible(), reason="fabricated device addresses: host-only test")


def _fwd(moe, cfg, **over):
    a = dict(x=FAKE, W_g=FAKE, W1=FAKE, W2=FAKE, W3=FAKE, y=FAKE, ws=FAKE, ws_bytes=1 << 40)
    a.update(over)
    ws_bytes = a.pop("ws_bytes")
    try:
        moe.forward(cfg, a.pop("x"), a.pop("W_g"), a.pop("W1"), a.pop("W2"), a.pop("W3"), a.pop("y"), a.pop("ws"),
                    ws_bytes=ws_bytes, stream=0, **a)
    except moe.MoEError as e:
        return e.status
    return moe.MOE_OK


@host_only
def test_argument_errors(moe):
    ok = moe.config(16, 64, 64, 8, 2)
    assert _fwd(moe, moe.config(16, 64, 64, 8, 9)) == moe.MOE_ERR_INVALID_ARG          # k > E
    assert _fwd(moe, moe.config(16, 0, 64, 8, 2)) == moe.MOE_ERR_INVALID_ARG           # d = 0
    assert _fwd(moe, moe.config(-1, 64, 64, 8, 2)) == moe.MOE_ERR_INVALID_ARG          # T < 0
    assert _fwd(moe, moe.config(16, 64, 64, 2000, 2)) == moe.MOE_ERR_UNSUPPORTED       # E > 1024
    assert _fwd(moe, moe.config(16, 64, 64, 64, 33)) == moe.MOE_ERR_UNSUPPORTED        # k > 32
    assert _fwd(moe, moe.config(16, 60, 64, 8, 2)) == moe.MOE_ERR_UNSUPPORTED          # bf16 d % 8
    assert _fwd(moe, ok, x=None) == moe.MOE_ERR_INVALID_ARG
    assert _fwd(moe, ok, x=FAKE + 2) == moe.MOE_ERR_INVALID_ARG                        # misaligned
    assert _fwd(moe, ok, W3=None) == moe.MOE_ERR_INVALID_ARG
    assert _fwd(moe, ok, ws=None) == moe.MOE_ERR_WORKSPACE
    assert _fwd(moe, ok, ws_bytes=moe.workspace_bytes(ok) - 1) == moe.MOE_ERR_WORKSPACE
    shared = moe.config(16, 64, 64, 8, 2, n_shared=1, d_ff_shared=64)
    assert _fwd(moe, shared) == moe.MOE_ERR_INVALID_ARG                                # Ws* missing
    bad_cfg = moe.config(16, 64, 64, 8, 2)
    bad_cfg.dtype = 7
    assert _fwd(moe, bad_cfg) == moe.MOE_ERR_INVALID_ARG
    bad_cfg = moe.config(16, 64, 64, 8, 2)
    bad_cfg.scoring = 5
    assert _fwd(moe, bad_cfg) == moe.MOE_ERR_INVALID_ARG
    for cf in (-1.0, float("nan"), float("inf")):
        assert _fwd(moe, moe.config(16, 64, 64, 8, 2, capacity_factor=cf)) == moe.MOE_ERR_INVALID_ARG


@host_only
def test_empty_batch_launches_nothing(moe):
    assert _fwd(moe, moe.config(0, 64, 64, 8, 2), ws_bytes=0) == moe.MOE_OK
    assert moe.last_launch_count() == 0


@host_only
def test_stage_argument_errors(moe):
    cfg = moe.config(16, 64, 64, 64, 4)   # E > 32: moe_route needs a workspace for the logits
    with pytest.raises(moe.MoEError) as e:
        moe.route(cfg, FAKE, FAKE, FAKE, FAKE, ws=None, stream=0)
    assert e.value.status == moe.MOE_ERR_WORKSPACE
    with pytest.raises(moe.MoEError) as e:
        moe.dispatch(cfg, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, ws_bytes=16, stream=0)
    assert e.value.status == moe.MOE_ERR_WORKSPACE
    with pytest.raises(moe.MoEError) as e:
        moe.experts(cfg, FAKE, FAKE, FAKE, FAKE, None, FAKE, FAKE, ws_bytes=1 << 30, stream=0)
    assert e.value.status == moe.MOE_ERR_INVALID_ARG
    with pytest.raises(moe.MoEError) as e:
        moe.combine(cfg, FAKE, FAKE, FAKE, None, stream=0)
    assert e.value.status == moe.MOE_ERR_INVALID_ARG


@host_only
def test_update_sel_bias_argument_errors(moe):
    cfg = moe.config(16, 64, 64, 8, 2)
    for counts, gamma, sb in ((None, 0.1, FAKE), (FAKE, 0.1, None), (FAKE + 2, 0.1, FAKE), (FAKE, -1.0, FAKE),
                              (FAKE, float("nan"), FAKE), (FAKE, float("inf"), FAKE)):
        with pytest.raises(moe.MoEError) as e:
            moe.update_sel_bias(cfg, counts, gamma, sb, stream=0)
        assert e.value.status == moe.MOE_ERR_INVALID_ARG
    with pytest.raises(moe.MoEError) as e:
        moe.update_sel_bias(moe.config(16, 64, 64, 8, 9), FAKE, 0.1, FAKE, stream=0)
    assert e.value.status == moe.MOE_ERR_INVALID_ARG


@host_only
def test_static_dispatch_rejects_sizes_beyond_its_array(moe):
    # ceil(T k / 256) * E = 513 * 256 = 131328 > 131072: refused before anything is launched
    cfg = moe.config(16384 + 32, 64, 64, 256, 8)
    with pytest.raises(moe.MoEError) as e:
        moe.dispatch_static(cfg, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, stream=0)
    assert e.value.status == moe.MOE_ERR_UNSUPPORTED


@host_only
def test_expert_choice_rejects_token_choice_calls(moe):
    cfg = moe.config(64, 64, 64, 8, 2, scoring="expert_choice")
    with pytest.raises(moe.MoEError) as e:
        moe.dispatch(cfg, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, ws_bytes=1 << 30, stream=0)
    assert e.value.status == moe.MOE_ERR_UNSUPPORTED
    with pytest.raises(moe.MoEError) as e:
        moe.dispatch_static(cfg, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, stream=0)
    assert e.value.status == moe.MOE_ERR_UNSUPPORTED
    assert _fwd(moe, cfg, topk_idx_out=FAKE) == moe.MOE_ERR_UNSUPPORTED
