"""Host-side checks of the C ABI that need no GPU: the library builds and
loads, exports every entry point ``include/ra.h`` declares, and rejects bad
arguments on the host before touching CUDA."""

import ctypes
import os
import re

import pytest

from long_context_exact_gb300 import binding

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "ra.h")


@pytest.fixture(scope="module")
def lib():
    from long_context_exact_gb300 import build as b
    b.build()
    return binding.load()


def _declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(ra_[a-z_0-9]+)\s*\(", text)))


def test_header_declares_the_boundary():
    names = _declared_functions()
    for required in ("ra_block_step", "ra_finalize", "ra_merge", "ra_ring_attention",
                     "ra_ring_attention_bwd", "ra_bwd_workspace_size", "ra_position_map",
                     "ra_ring_order", "ra_stream_check", "ra_last_error"):
        assert required in names


def test_library_exports_every_declared_symbol(lib):
    for name in _declared_functions():
        assert hasattr(lib, name), name


def test_version(lib):
    assert lib.ra_version() >= 100


def _dims(b=1, h=4, n_kv=2, d=128):
    return binding.Dims(b, h, n_kv, d)


FAKE = ctypes.c_void_p(0x10000)      # aligned, never dereferenced: calls fail earlier
MISALIGNED = ctypes.c_void_p(0x10008)


@pytest.mark.parametrize("dims,status", [
    (dict(d=96), binding.RA_ERR_UNSUPPORTED),
    (dict(h=6, n_kv=4), binding.RA_ERR_UNSUPPORTED),
    (dict(h=0), binding.RA_ERR_INVALID_ARG),
    (dict(b=-1), binding.RA_ERR_INVALID_ARG),
])
def test_ring_attention_rejects_bad_dims(lib, dims, status):
    st = lib.ra_ring_attention(FAKE, FAKE, FAKE, FAKE, FAKE, 1024, 4, 1, 1, 0.0, _dims(**dims), None)
    assert st == status
    assert lib.ra_last_error()


def test_ring_attention_rejects_bad_sizes_and_pointers(lib):
    d = _dims()
    assert lib.ra_ring_attention(FAKE, FAKE, FAKE, FAKE, FAKE, 1000, 3, 1, 1, 0.0, d, None) == \
        binding.RA_ERR_UNSUPPORTED                      # S % N != 0
    assert lib.ra_ring_attention(FAKE, FAKE, FAKE, FAKE, FAKE, 1024, 0, 1, 1, 0.0, d, None) == \
        binding.RA_ERR_INVALID_ARG                      # N < 1
    assert lib.ra_ring_attention(FAKE, FAKE, FAKE, FAKE, FAKE, 1024, 4, 7, 1, 0.0, d, None) == \
        binding.RA_ERR_INVALID_ARG                      # layout
    assert lib.ra_ring_attention(None, FAKE, FAKE, FAKE, FAKE, 1024, 4, 1, 1, 0.0, d, None) == \
        binding.RA_ERR_INVALID_ARG                      # null q
    assert "q" in lib.ra_last_error().decode()
    assert lib.ra_ring_attention(FAKE, MISALIGNED, FAKE, FAKE, FAKE, 1024, 4, 1, 1, 0.0, d, None) == \
        binding.RA_ERR_INVALID_ARG                      # misaligned k
    assert lib.ra_ring_attention(FAKE, FAKE, FAKE, FAKE, FAKE, 1024, 4, 1, 1, float("nan"), d,
                                 None) == binding.RA_ERR_INVALID_ARG
    assert lib.ra_ring_attention(FAKE, FAKE, FAKE, FAKE, FAKE, 1 << 31, 1, 1, 1, 0.0, d, None) == \
        binding.RA_ERR_UNSUPPORTED


def test_empty_inputs_are_a_no_op(lib):
    d = _dims()
    assert lib.ra_ring_attention(None, None, None, None, None, 0, 4, 1, 1, 0.0, d, None) == binding.RA_OK
    assert lib.ra_ring_attention(None, None, None, None, None, 512, 4, 1, 1, 0.0, _dims(b=0),
                                 None) == binding.RA_OK
    assert lib.ra_block_step(None, None, None, None, None, None, None, None, 0, 128, d, 1, 0.0,
                             None) == binding.RA_OK
    assert lib.ra_finalize(None, None, None, None, 0, d, None) == binding.RA_OK
    assert lib.ra_merge(None, None, None, None, None, None, 0, d, None) == binding.RA_OK


def test_block_step_validation(lib):
    d = _dims()
    assert lib.ra_block_step(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, None, None, 128, 128, d, 1, 0.0,
                             None) == binding.RA_ERR_INVALID_ARG   # causal without positions
    assert lib.ra_block_step(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, None, None, -1, 128, d, 0, 0.0,
                             None) == binding.RA_ERR_INVALID_ARG


def test_map_and_order_validation(lib):
    assert lib.ra_position_map(1, 1000, 3, FAKE, FAKE, FAKE, None) == binding.RA_ERR_UNSUPPORTED
    assert lib.ra_position_map(5, 1024, 4, FAKE, FAKE, FAKE, None) == binding.RA_ERR_INVALID_ARG
    assert lib.ra_ring_order(0, FAKE, None) == binding.RA_ERR_INVALID_ARG
    assert lib.ra_ring_order(4, None, None) == binding.RA_ERR_INVALID_ARG
    assert lib.ra_selftest_wait_timeout(0, None) == binding.RA_ERR_INVALID_ARG


def test_zigzag_shape_validation(lib):
    d = _dims()
    # half-blocks must be whole 128-token tiles for the attention calls
    assert lib.ra_ring_attention(FAKE, FAKE, FAKE, FAKE, FAKE, 1024, 8, 2, 1, 0.0, d, None) == \
        binding.RA_ERR_UNSUPPORTED                      # S / 2N = 64
    assert "zig-zag" in lib.ra_last_error().decode()
    assert lib.ra_ring_attention(FAKE, FAKE, FAKE, FAKE, FAKE, 1536, 4, 2, 1, 0.0, d, None) == \
        binding.RA_ERR_UNSUPPORTED                      # S / 2N = 192
    assert lib.ra_ring_attention_bwd(*([FAKE] * 9), FAKE, 1 << 30, 1024, 8, 2, 1, 0.0, d,
                                     None) == binding.RA_ERR_UNSUPPORTED
    assert lib.ra_ring_attention_bwd_noalloc(*([FAKE] * 9), 1024, 8, 2, 1, 0.0, d,
                                             None) == binding.RA_ERR_UNSUPPORTED
    # the maps only need an even split into 2N half-blocks
    assert lib.ra_position_map(2, 12, 4, FAKE, FAKE, FAKE, None) == binding.RA_ERR_UNSUPPORTED
    assert lib.ra_position_map(3, 16, 4, FAKE, FAKE, FAKE, None) == binding.RA_ERR_INVALID_ARG


def test_ex2_probe_validation(lib):
    n = lib.ra_ex2_probe_threads()
    assert n > 0 and n % 256 == 0
    assert lib.ra_ex2_probe(0, FAKE, n, None) == binding.RA_ERR_INVALID_ARG
    assert lib.ra_ex2_probe(16, None, n, None) == binding.RA_ERR_INVALID_ARG
    assert lib.ra_ex2_probe(16, FAKE, n - 1, None) == binding.RA_ERR_INVALID_ARG


def test_prefill_validation_and_workspace(lib):
    lib.ra_prefill_workspace_size.argtypes = [ctypes.c_int64, ctypes.c_int64, ctypes.c_int,
                                              binding.Dims]
    lib.ra_prefill_workspace_size.restype = ctypes.c_size_t
    d = _dims(b=1, h=8, n_kv=2, d=128)
    # explicit split counts: n_splits states of (m, l, O) per query row, then
    # one int per 128-query tile and one per 128-key tile (each rounded up to
    # 16 bytes)
    def size(splits, Lq=256, Lk=4096):
        return (splits * 8 * Lq * (2 + 128) * 4 + ((Lq + 127) // 128 * 4 + 15) // 16 * 16 +
                ((Lk + 127) // 128 * 4 + 15) // 16 * 16)
    assert lib.ra_prefill_workspace_size(256, 4096, 4, d) == size(4)
    # never more splits than key tiles, and no empty split
    assert lib.ra_prefill_workspace_size(256, 300, 8, d) == size(3, Lk=300)
    assert lib.ra_prefill_workspace_size(256, 1280, 4, d) == size(4, Lk=1280)
    assert lib.ra_prefill_workspace_size(256, 1280, 6, d) == size(5, Lk=1280)
    assert lib.ra_prefill_workspace_size(0, 4096, 4, d) == 0
    args = [FAKE] * 7
    assert lib.ra_chunked_prefill(*args, 256, 4096, 65, d, 1, 0.0, FAKE, 1 << 30, None) == \
        binding.RA_ERR_INVALID_ARG                      # too many splits
    assert lib.ra_chunked_prefill(*args[:5], None, None, 256, 4096, 0, d, 1, 0.0, FAKE, 1 << 30,
                                  None) == binding.RA_ERR_INVALID_ARG   # causal without positions
    assert lib.ra_chunked_prefill(*args, 256, 4096, 4, d, 1, 0.0, None, 0, None) == \
        binding.RA_ERR_WORKSPACE
    assert lib.ra_chunked_prefill(*args, 256, 4096, 4, d, 1, 0.0, FAKE, 16, None) == \
        binding.RA_ERR_WORKSPACE
    assert lib.ra_chunked_prefill(*args, 0, 4096, 4, d, 1, 0.0, None, 0, None) == binding.RA_OK


def test_packed_validation(lib):
    d = _dims()
    assert lib.ra_ring_attention_packed(FAKE, FAKE, FAKE, FAKE, FAKE, 1024, 4, 1, 1, 0.0, d, FAKE,
                                        0, None) == binding.RA_ERR_INVALID_ARG   # no documents
    assert lib.ra_ring_attention_packed(FAKE, FAKE, FAKE, FAKE, FAKE, 1024, 4, 1, 1, 0.0, d, None,
                                        3, None) == binding.RA_ERR_INVALID_ARG   # offsets missing
    assert lib.ra_ring_attention_packed_bwd(*([FAKE] * 9), FAKE, 1 << 30, 1024, 4, 1, 1, 0.0, d,
                                            FAKE, -1, None) == binding.RA_ERR_INVALID_ARG


def test_workspace_size(lib):
    lib.ra_bwd_workspace_size.argtypes = [ctypes.c_int64, ctypes.c_int, binding.Dims]
    n = lib.ra_bwd_workspace_size(65536, 16, _dims(b=2, h=32, n_kv=8))
    assert n == 2 * 2 * 32 * 65536 * 4
    # rows of each shard are padded to a multiple of 128
    assert lib.ra_bwd_workspace_size(600, 3, _dims(b=1, h=4)) == 2 * 4 * 3 * 256 * 4
    assert lib.ra_bwd_workspace_size(0, 4, _dims()) == 0
    assert lib.ra_bwd_workspace_size(1000, 3, _dims()) == 0


def test_bwd_validation(lib):
    d = _dims()
    args = [FAKE] * 9
    assert lib.ra_ring_attention_bwd(*args, None, 0, 1024, 4, 1, 1, 0.0, d, None) == \
        binding.RA_ERR_WORKSPACE
    assert lib.ra_ring_attention_bwd(*args, FAKE, 16, 1024, 4, 1, 1, 0.0, d, None) == \
        binding.RA_ERR_WORKSPACE
    assert lib.ra_ring_attention_bwd(*args, FAKE, 1 << 30, 1024, 4, 1, 1, 0.0, _dims(d=80),
                                     None) == binding.RA_ERR_UNSUPPORTED
    bad = list(args)
    bad[5] = None
    assert lib.ra_ring_attention_bwd(*bad, FAKE, 1 << 30, 1024, 4, 1, 1, 0.0, d, None) == \
        binding.RA_ERR_INVALID_ARG


def test_binding_refuses_cpu_tensors(lib):
    import torch
    q = torch.zeros((1, 128, 2, 64), dtype=torch.bfloat16)
    with pytest.raises(binding.RAError):
        binding.ring_attention(q, q, q, 1)


def test_host_buffer_and_pipeline_validation(lib):
    """Argument checks of the host-buffer calls, all before any CUDA call."""
    P = ctypes.c_void_p
    out = P()
    assert lib.ra_host_alloc(0, ctypes.byref(out)) == binding.RA_OK and out.value is None
    assert lib.ra_host_alloc(16, None) == binding.RA_ERR_INVALID_ARG
    assert lib.ra_host_free(None) == binding.RA_OK
    h = P()
    create = lib.ra_pipeline_create
    assert create(1024, 4, 1, 1, 0.0, _dims(), 1, None) == binding.RA_ERR_INVALID_ARG
    assert create(0, 4, 1, 1, 0.0, _dims(), 1, ctypes.byref(h)) == binding.RA_ERR_INVALID_ARG
    assert create(1024, 0, 1, 1, 0.0, _dims(), 1, ctypes.byref(h)) == binding.RA_ERR_INVALID_ARG
    assert create(8, 16, 1, 1, 0.0, _dims(), 1, ctypes.byref(h)) == binding.RA_ERR_INVALID_ARG
    assert create(1024, 4, 1, 1, 0.0, _dims(d=96), 1, ctypes.byref(h)) == \
        binding.RA_ERR_UNSUPPORTED
    assert create(1024, 4, 1, 1, 0.0, _dims(h=6, n_kv=4), 1, ctypes.byref(h)) == \
        binding.RA_ERR_UNSUPPORTED
    assert create(1024, 4, 7, 1, 0.0, _dims(), 1, ctypes.byref(h)) == binding.RA_ERR_INVALID_ARG
    assert h.value is None
    assert lib.ra_pipeline_submit(None, FAKE, FAKE, FAKE, FAKE, None, None, None, None,
                                  None) == binding.RA_ERR_INVALID_ARG
    assert lib.ra_pipeline_sync(None) == binding.RA_ERR_INVALID_ARG
    assert lib.ra_pipeline_destroy(None) == binding.RA_OK


def test_causal_block_ranges_are_bounded(lib):
    """A causal block step classifies its whole key range in shared memory:
    at most 65,536 key tiles (8,388,608 keys); longer ranges are refused on
    the host, and a chunked prefill needs enough key splits."""
    d = _dims()
    over = 65536 * 128 + 1
    assert lib.ra_block_step(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 128, over, d, 1,
                             0.0, None) == binding.RA_ERR_UNSUPPORTED
    assert b"at most 8388608 keys" in lib.ra_last_error()
    lib.ra_prefill_workspace_size.argtypes = [ctypes.c_int64, ctypes.c_int64, ctypes.c_int,
                                              binding.Dims]
    lib.ra_prefill_workspace_size.restype = ctypes.c_size_t
    st = lib.ra_chunked_prefill(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 128, 2 * over, 1, d, 1,
                                0.0, FAKE, 1 << 40, None)
    assert st == binding.RA_ERR_UNSUPPORTED
    # the automatic split count covers long ranges
    rows = 1 * 4 * 128
    need = lib.ra_prefill_workspace_size(128, 2 * over, 0, d)
    assert need >= 3 * rows * (2 + 128) * 4


def test_block_step_bwd_validates_on_the_host(lib):
    """The block backward rejects bad arguments before any launch: causal
    without positions, a missing or short workspace, null or misaligned
    pointers; empty blocks are a no-op."""
    d = _dims()
    ws = lib.ra_block_bwd_workspace_size(1024, d)
    assert ws == lib.ra_bwd_workspace_size(1024, 1, d) == 2 * 1 * 4 * 1024 * 4
    args = [FAKE] * 9
    # causal without q_pos / k_pos
    assert lib.ra_block_step_bwd(*args, None, None, 1024, 512, d, 1, 0.0, FAKE, ws, None) == \
        binding.RA_ERR_INVALID_ARG
    # workspace missing or too small
    assert lib.ra_block_step_bwd(*args, FAKE, FAKE, 1024, 512, d, 1, 0.0, None, 0, None) == \
        binding.RA_ERR_WORKSPACE
    assert lib.ra_block_step_bwd(*args, FAKE, FAKE, 1024, 512, d, 1, 0.0, FAKE, ws - 16,
                                 None) == binding.RA_ERR_WORKSPACE
    # null dk, misaligned dout
    bad = list(args)
    bad[7] = None
    assert lib.ra_block_step_bwd(*bad, FAKE, FAKE, 1024, 512, d, 1, 0.0, FAKE, ws, None) == \
        binding.RA_ERR_INVALID_ARG
    assert "dk" in lib.ra_last_error().decode()
    bad = list(args)
    bad[5] = MISALIGNED
    assert lib.ra_block_step_bwd(*bad, FAKE, FAKE, 1024, 512, d, 1, 0.0, FAKE, ws, None) == \
        binding.RA_ERR_INVALID_ARG
    # d unsupported, negative length
    assert lib.ra_block_step_bwd(*args, FAKE, FAKE, 1024, 512, _dims(d=96), 1, 0.0, FAKE, ws,
                                 None) == binding.RA_ERR_UNSUPPORTED
    assert lib.ra_block_step_bwd(*args, FAKE, FAKE, -1, 512, d, 1, 0.0, FAKE, ws, None) == \
        binding.RA_ERR_INVALID_ARG
    # empty blocks: nothing to do, nothing launched
    assert lib.ra_block_step_bwd(*args, FAKE, FAKE, 0, 512, d, 1, 0.0, None, 0, None) == \
        binding.RA_OK
    assert lib.ra_block_step_bwd(*args, FAKE, FAKE, 1024, 0, d, 1, 0.0, None, 0, None) == \
        binding.RA_OK
