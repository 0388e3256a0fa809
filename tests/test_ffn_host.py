"""The blockwise feed-forward entry points of include/ring_attn.h on the
host (no GPU): workspace size and the argument checks that return before
anything is launched."""
import ctypes

import pytest

from sequence_blockwise_self_gb300 import build as lib_build
from sequence_blockwise_self_gb300 import capi

P256 = ctypes.c_void_p(256)   # an aligned, never dereferenced address
P8 = ctypes.c_void_p(264)     # 8-byte but not 16-byte aligned
NUL = ctypes.c_void_p(0)


@pytest.fixture(scope="module")
def lib():
    lib_build.build()
    return capi.load()


def test_workspace_is_one_hidden_block(lib):
    # the BPT saving: one block of the hidden activation, bf16
    assert lib.ring_attn_ffn_workspace_size(3584, 14336, 8192) == 8192 * 14336 * 2
    assert lib.ring_attn_ffn_workspace_size(256, 768, 128) == 128 * 768 * 2


@pytest.mark.parametrize("D,F,R", [(256, 1000, 128), (300, 1024, 128), (256, 1024, 100), (0, 1024, 128),
                                   (256, 1024, 0), (256, -256, 128)])
def test_unsupported_shapes_have_no_workspace(lib, D, F, R):
    assert lib.ring_attn_ffn_workspace_size(D, F, R) == 0


def test_argument_errors(lib):
    ws = lib.ring_attn_ffn_workspace_size(256, 1024, 256)
    ptrs = [P256] * 6
    f = lib.ring_attn_ffn_fwd
    assert f(*ptrs, -1, 256, 1024, 256, P256, ws, NUL) == capi.ERR_SHAPE
    assert f(*ptrs, 1 << 31, 256, 1024, 256, P256, ws, NUL) == capi.ERR_UNSUPPORTED
    assert f(*ptrs, 1000, 200, 1024, 256, P256, ws, NUL) == capi.ERR_UNSUPPORTED
    assert f(*ptrs, 1000, 256, 1024, 0, P256, ws, NUL) == capi.ERR_SHAPE
    assert f(*([NUL] * 6), 1000, 256, 1024, 256, P256, ws, NUL) == capi.ERR_NULL
    for i in range(6):
        args = list(ptrs)
        args[i] = P8
        assert f(*args, 1000, 256, 1024, 256, P256, ws, NUL) == capi.ERR_UNSUPPORTED
    assert f(*ptrs, 1000, 256, 1024, 256, NUL, ws, NUL) == capi.ERR_WORKSPACE
    assert f(*ptrs, 1000, 256, 1024, 256, P256, ws - 1, NUL) == capi.ERR_WORKSPACE
    assert f(*ptrs, 1000, 256, 1024, 256, ctypes.c_void_p(256 + 16), ws, NUL) == capi.ERR_WORKSPACE


def test_empty_input_is_a_no_op(lib):
    assert lib.ring_attn_ffn_fwd(*([NUL] * 6), 0, 256, 1024, 256, NUL, 0, NUL) == capi.OK


def test_bpt_workspace_and_argument_errors(lib):
    assert lib.ring_attn_bpt_workspace_size(28, 128, 14336, 8192) == 8192 * 14336 * 2
    assert lib.ring_attn_bpt_workspace_size(28, 128, 14336, 128) == 0   # not whole 256-row work items
    f = lib.ring_attn_bpt_fwd
    ws = lib.ring_attn_bpt_workspace_size(2, 128, 1024, 256)
    ptrs = [P256] * 10
    # (B, Hq, Hkv, L, d, N, causal, F, block_rows)
    assert f(*ptrs, 1, 2, 1, 1024, 128, 4, 1, 1024, 128, P256, ws, NUL) == capi.ERR_UNSUPPORTED
    assert f(*ptrs, 1, 2, 1, 1024, 128, 4, 1, 1024, 0, P256, ws, NUL) == capi.ERR_SHAPE
    assert f(*ptrs, 1, 3, 1, 1024, 128, 4, 1, 1024, 256, P256, ws, NUL) == capi.ERR_UNSUPPORTED  # D = 384
    assert f(*ptrs, 1, 2, 1, 1024, 128, 4, 1, 1000, 256, P256, ws, NUL) == capi.ERR_UNSUPPORTED  # F % 256
    assert f(*ptrs, 1, 2, 1, 1004, 128, 4, 1, 1024, 256, P256, ws, NUL) == capi.ERR_SHAPE  # causal L % 2N
    assert f(*([NUL] * 10), 1, 2, 1, 1024, 128, 4, 1, 1024, 256, P256, ws, NUL) == capi.ERR_NULL
    assert f(*ptrs, 1, 2, 1, 1024, 128, 4, 1, 1024, 256, P256, ws - 1, NUL) == capi.ERR_WORKSPACE
    args = list(ptrs)
    args[3] = P8
    assert f(*args, 1, 2, 1, 1024, 128, 4, 1, 1024, 256, P256, ws, NUL) == capi.ERR_UNSUPPORTED
    assert f(*([NUL] * 10), 0, 2, 1, 1024, 128, 4, 1, 1024, 256, NUL, 0, NUL) == capi.OK   # B == 0


def test_ffn_bwd_and_bpt_bwd_arguments(lib):
    assert lib.ring_attn_ffn_bwd_workspace_size(256, 512, 128) > 0
    assert lib.ring_attn_ffn_bwd_workspace_size(200, 512, 128) == 0
    ws = lib.ring_attn_ffn_bwd_workspace_size(256, 512, 128)
    f = lib.ring_attn_ffn_bwd
    ptrs = [P256] * 10
    assert f(*ptrs, -1, 256, 512, 128, P256, ws, NUL) == capi.ERR_SHAPE
    assert f(*([NUL] * 10), 100, 256, 512, 128, P256, ws, NUL) == capi.ERR_NULL
    assert f(*ptrs, 100, 256, 512, 128, P256, ws - 1, NUL) == capi.ERR_WORKSPACE
    assert f(*ptrs, 100, 256, 512, 100, P256, ws, NUL) == capi.ERR_UNSUPPORTED
    g = lib.ring_attn_bpt_bwd
    wsb = lib.ring_attn_bpt_bwd_workspace_size(1, 2, 1, 1024, 128, 4, 1, 1024, 256)
    assert wsb > ws
    assert lib.ring_attn_bpt_bwd_workspace_size(1, 2, 1, 1024, 128, 4, 1, 1024, 128) == 0
    bptrs = [P256] * 16
    assert g(*bptrs, 1, 2, 1, 1024, 128, 4, 1, 1024, 128, P256, wsb, NUL) == capi.ERR_UNSUPPORTED
    assert g(*([NUL] * 16), 1, 2, 1, 1024, 128, 4, 1, 1024, 256, P256, wsb, NUL) == capi.ERR_NULL
    assert g(*bptrs, 1, 2, 1, 1024, 128, 4, 1, 1024, 256, P256, wsb - 1, NUL) == capi.ERR_WORKSPACE


def test_every_pointer_must_be_16_byte_aligned(lib):
    """The kernels read every operand with 16-byte accesses (TMA boxes, and
    the biases by 16-byte copies into shared memory), so each pointer of the
    FFN and BPT entries that is not 16-byte aligned is refused before any
    device work."""
    ws = lib.ring_attn_ffn_bwd_workspace_size(256, 512, 128)
    for i in range(10):
        args = [P256] * 10
        args[i] = P8
        assert lib.ring_attn_ffn_bwd(*args, 100, 256, 512, 128, P256, ws, NUL) == capi.ERR_UNSUPPORTED, i
    ws = lib.ring_attn_bpt_workspace_size(2, 128, 1024, 256)
    for i in range(10):
        args = [P256] * 10
        args[i] = P8
        assert lib.ring_attn_bpt_fwd(*args, 1, 2, 1, 1024, 128, 4, 1, 1024, 256, P256, ws, NUL) == \
            capi.ERR_UNSUPPORTED, i
    wsb = lib.ring_attn_bpt_bwd_workspace_size(1, 2, 1, 1024, 128, 4, 1, 1024, 256)
    for i in range(16):
        args = [P256] * 16
        args[i] = P8
        assert lib.ring_attn_bpt_bwd(*args, 1, 2, 1, 1024, 128, 4, 1, 1024, 256, P256, wsb, NUL) == \
            capi.ERR_UNSUPPORTED, i
