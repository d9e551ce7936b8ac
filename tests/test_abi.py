"""The C-ABI library builds, loads and exports what its header declares, and
its host-side argument checks answer before anything reaches a GPU (CPU)."""
import ctypes

import pytest

from target_model_verify_gb300 import _binding as b
from target_model_verify_gb300 import build as libbuild


@pytest.fixture(scope="module")
def lib():
    libbuild.build()
    return b.lib()


def test_exports_every_header_symbol(lib):
    names = b.header_functions()
    assert len(names) >= 9
    for name in names:
        assert hasattr(lib, name), name
    assert set(names) == set(b._SIGNATURES)


def test_status_strings(lib):
    for code in (0, -1, -2, -3, -4, -5, -6):
        assert b.status_string(code) not in ("", "unknown status")
    assert b.status_string(-99) == "unknown status"


def test_workspace_size(lib):
    n = b.specdec_verify_workspace_size(1, 4, 4096, 128256, b.SPECDEC_BF16, b.SPECDEC_SAMPLE)
    # holds at least the fp32 logits of the 5 rows
    assert n >= 5 * 128256 * 4
    g = b.specdec_verify_workspace_size(1, 4, 4096, 128256, b.SPECDEC_BF16, b.SPECDEC_GREEDY)
    assert 0 < g < n
    assert b.specdec_verify_workspace_size(1, 0, 4096, 128256, 0, 0) == 0      # gamma = 0
    assert b.specdec_verify_workspace_size(1, 33, 4096, 128256, 0, 0) == 0     # gamma > max
    assert b.specdec_verify_workspace_size(1, 4, 4090, 128256, 0, 0) == 0      # d % 8 != 0
    assert b.specdec_verify_workspace_size(1, 4, 64, 512, 7, 0) == 0          # bad dtype
    assert b.specdec_verify_workspace_size(1, 4, 64, 512, 0, 3) == 0          # bad mode
    assert b.specdec_verify_workspace_size(20000, 32, 64, 128256, 0, 0) == 0  # M*V >= 2^31
    h = b.specdec_verify_host_workspace_size(1, 4, 4096, 128256, 0, 0)
    assert h > n


def _call(B=1, gamma=4, d=64, V=512, dtype=1, T=1.0, mode=0, ptr=4096, ws=256, ws_bytes=1 << 30,
          dl=4096):
    # Fake but aligned addresses: every check below fails before any access.
    return b.specdec_verify(ptr, ptr, ptr, dl, B, gamma, d, V, dtype, T, 0, mode, ptr, ptr,
                            ws, ws_bytes, None)


def test_host_side_argument_errors(lib):
    assert _call(ptr=0) == b.SPECDEC_ERR_INVALID_ARG
    assert _call(dl=0) == b.SPECDEC_ERR_INVALID_ARG                 # sampling needs q
    assert _call(T=0.0) == b.SPECDEC_ERR_INVALID_ARG
    assert _call(T=-1.0) == b.SPECDEC_ERR_INVALID_ARG
    assert _call(T=float("nan")) == b.SPECDEC_ERR_INVALID_ARG
    assert _call(gamma=0) == b.SPECDEC_ERR_UNSUPPORTED
    assert _call(gamma=33) == b.SPECDEC_ERR_UNSUPPORTED
    assert _call(dtype=0, d=60) == b.SPECDEC_ERR_UNSUPPORTED
    assert _call(dtype=0, ptr=4098) == b.SPECDEC_ERR_INVALID_ARG     # bf16 needs 16B alignment
    assert _call(ws=0) == b.SPECDEC_ERR_WORKSPACE
    assert _call(ws=300) == b.SPECDEC_ERR_WORKSPACE                  # misaligned
    assert _call(ws_bytes=16) == b.SPECDEC_ERR_WORKSPACE
    assert _call(B=0) == b.SPECDEC_OK                                # empty batch: no-op
    assert _call(mode=5) == b.SPECDEC_ERR_INVALID_ARG
    # greedy mode does not need draft logits or a temperature
    assert _call(mode=1, dl=0, T=0.0, ws=0) == b.SPECDEC_ERR_WORKSPACE


def test_philox_argument_errors(lib):
    assert b.specdec_philox_uniforms(0, 1, 1, 2, 4096, None) == b.SPECDEC_ERR_INVALID_ARG
    assert b.specdec_philox_uniforms(0, 1, 1, 0, 0, None) == b.SPECDEC_ERR_INVALID_ARG
    assert b.specdec_philox_uniforms(0, 0, 5, 0, 4096, None) == b.SPECDEC_OK


def test_read_status_argument_errors(lib):
    st = ctypes.c_int32(0)
    assert lib.specdec_read_status(None, None, ctypes.byref(st)) == b.SPECDEC_ERR_INVALID_ARG


def _tree_call(parent=(-1, 0, 0, 1), B=1, d=64, V=512, dtype=0, T=1.0, mode=0, ptr=4096, ws=256,
               ws_bytes=1 << 30, dl=4096):
    par = (ctypes.c_int32 * max(1, len(parent)))(*parent)
    N = len(parent)
    return b.specdec_verify_tree(ptr, ptr, ctypes.addressof(par), ptr, dl, B, N, d, V, dtype, T,
                                 0, mode, ptr, ptr, ptr, ws, ws_bytes, 0)


def test_tree_workspace_and_host_side_errors(lib):
    n = b.specdec_verify_tree_workspace_size(2, 26, 64, 1000, 0, 0)
    g = b.specdec_verify_tree_workspace_size(2, 26, 64, 1000, 0, 1)
    assert n > g > 0                                   # sampling keeps logits and q records
    assert b.specdec_verify_tree_workspace_size(2, 129, 64, 1000, 0, 0) == 0   # > max nodes
    assert b.specdec_verify_tree_workspace_size(2, 26, 64, 1000, 1, 0) == 0    # fp32: no tree path
    assert _tree_call(parent=(0, 0)) == b.SPECDEC_ERR_INVALID_ARG              # root not -1
    assert _tree_call(parent=(-1, 1)) == b.SPECDEC_ERR_INVALID_ARG             # self parent
    assert _tree_call(parent=(-1, 0, 3, 0)) == b.SPECDEC_ERR_INVALID_ARG       # later parent
    assert _tree_call(dtype=1) == b.SPECDEC_ERR_UNSUPPORTED
    assert _tree_call(dl=0) == b.SPECDEC_ERR_INVALID_ARG                       # sampling needs q
    assert _tree_call(T=0.0) == b.SPECDEC_ERR_INVALID_ARG
    assert _tree_call(ptr=4098) == b.SPECDEC_ERR_INVALID_ARG                   # 16-byte alignment
    assert _tree_call(ws=0) == b.SPECDEC_ERR_WORKSPACE
    assert _tree_call(ws_bytes=16) == b.SPECDEC_ERR_WORKSPACE
    assert _tree_call(B=0) == b.SPECDEC_OK
    assert _tree_call(mode=1, dl=0, T=0.0, ws=0) == b.SPECDEC_ERR_WORKSPACE    # greedy: no q, no T


def test_shard_sizes_and_host_side_argument_errors(lib):
    """The vocabulary-parallel calls check their arguments on the host."""
    assert b.specdec_shard_record_bytes(256, 4) >= 256 * 5 * 16 + 256 * 4 * (8 + 16)
    assert b.specdec_shard_record_bytes(1, 0) == 0
    assert b.specdec_shard_workspace_size(1, 4, 4096, 32064, 0) > 5 * 32064 * 4
    assert b.specdec_shard_workspace_size(1, 4, 4090, 32064, 0) == 0     # d % 8 != 0
    ws, ptr = 4096 * 256, 4096
    big = 1 << 30
    # score: the slice must sit inside [0, V); temperature must be positive
    assert b.specdec_shard_score(ptr, ptr, ptr, ptr, 1, 4, 64, 500, 600, 1000, 1.0, 0, ptr, ws, big,
                                 None) == b.SPECDEC_ERR_UNSUPPORTED
    assert b.specdec_shard_score(ptr, ptr, ptr, ptr, 1, 4, 64, 500, 0, 1000, 0.0, 0, ptr, ws, big,
                                 None) == b.SPECDEC_ERR_INVALID_ARG
    assert b.specdec_shard_score(ptr, ptr, ptr, ptr, 1, 4, 64, 500, 0, 1000, 1.0, 0, ptr, 300, big,
                                 None) == b.SPECDEC_ERR_WORKSPACE
    # accept: 1 <= n_shards <= SPECDEC_MAX_SHARDS
    for n in (0, 65):
        assert b.specdec_shard_accept(ptr, n, ptr, ptr, 1, 4, 64, 500, 0, 1000, 1.0, 0, 0, ptr, ptr,
                                      ptr, ws, big, None) == b.SPECDEC_ERR_INVALID_ARG
    # draw: the caller's slice index must be one of the n_shards
    assert b.specdec_shard_draw(ptr, 2, 2, ptr, 1, 4, 64, 500, 0, 1000, 1.0, 0, 0, ptr, ws, big,
                                None) == b.SPECDEC_ERR_INVALID_ARG
    assert b.specdec_shard_draw(ptr, 2, -1, ptr, 1, 4, 64, 500, 0, 1000, 1.0, 0, 0, ptr, ws, big,
                                None) == b.SPECDEC_ERR_INVALID_ARG
    # greedy mode has nothing to draw: the call is a no-op
    assert b.specdec_shard_draw(0, 0, 0, 0, 1, 4, 64, 500, 0, 1000, 1.0, 0, 1, 0, ws, big,
                                None) == b.SPECDEC_OK


def test_bench_launch_count_follows_the_library_plan():
    """bench.py reports gpu_launches from its own copy of the launch plan
    (two kernels while B * chunks fits the fused acceptance-and-draw kernel,
    three up to the one-kernel sampler's limit, else four). Its thresholds
    must be the library's, read here from the kernel sources."""
    import os
    import re
    import bench
    from target_model_verify_gb300 import workloads as wl
    csrc = os.path.join(os.path.dirname(libbuild.__file__), "csrc")
    text = "".join(open(os.path.join(csrc, f)).read() for f in ("common.cuh", "kernels.h"))

    def constant(name):
        m = re.search(r"constexpr\s+(?:long\s+long|int)\s+%s\s*=\s*(\d+)\s*;" % name, text)
        assert m, name
        return int(m.group(1))

    assert bench.SAMPLE_CHUNK == constant("kChunkV")
    assert bench.FUSED_ITEMS == constant("kFusedAcceptItems")
    assert bench.ONE_DRAW_KERNEL_ITEMS == constant("kSampleOneKernelItems")
    expect = {"llama3_8b_head": 2, "llama3_8b_head_b4": 2, "llama3_8b_head_b16": 3,
              "llama3_8b_head_b64": 4, "llama3_8b_head_b256": 4, "head_70b_b32_g7": 4,
              "gemma_e2b_head_g1": 2}
    for name, n in expect.items():
        assert bench.kernels_per_step(wl.get(name), wl.SAMPLE) == n, name
        assert bench.kernels_per_step(wl.get(name), wl.GREEDY) == 2, name
