"""specdec_verify_noalloc: the verify step for callers that cannot allocate.

Some callers of this library cannot give it a workspace: code running inside
a host program that owns all device memory and offers plug-ins no
allocator, or a decode loop whose memory was planned up front, where a
cudaMalloc would synchronise the device or fail against a caching
allocator's reservation. For them the library keeps a fixed static scratch
array on each device. These tests call that entry point through the C ABI
and check it gives the same tokens as the workspace entry point, on two
calls in a row (the array keeps the previous call's contents), and that it
refuses shapes whose scratch would not fit.
"""
import numpy as np
import pytest
import torch

from target_model_verify_gb300 import _binding as b
from target_model_verify_gb300 import workloads as wl

SCRATCH_BYTES = 16 << 20


def _noalloc(inp, T, seed, mode, out, nacc, dl=None):
    B, g1, d = inp["hidden"].shape
    V = inp["W_lm"].shape[0]
    dtype = b.SPECDEC_BF16 if inp["hidden"].dtype == torch.bfloat16 else b.SPECDEC_FP32
    return b.specdec_verify_noalloc(
        inp["hidden"].data_ptr(), inp["W_lm"].data_ptr(), inp["draft_tokens"].data_ptr(),
        0 if dl is None else dl.data_ptr(), B, g1 - 1, d, V, dtype, T, seed, mode,
        out.data_ptr(), nacc.data_ptr(), torch.cuda.current_stream().cuda_stream)


def test_noalloc_rejects_shapes_beyond_its_scratch():
    """The size check answers on the host, before any pointer is used."""
    from target_model_verify_gb300 import build
    build.build()
    need = b.specdec_verify_workspace_size(64, 4, 4096, 128256, b.SPECDEC_BF16, b.SPECDEC_SAMPLE)
    assert need > SCRATCH_BYTES
    rc = b.specdec_verify_noalloc(4096, 4096, 4096, 4096, 64, 4, 4096, 128256, b.SPECDEC_BF16,
                                  1.0, 0, b.SPECDEC_SAMPLE, 4096, 4096, None)
    assert rc == b.SPECDEC_ERR_WORKSPACE
    # an invalid shape still reports the shape error
    rc = b.specdec_verify_noalloc(4096, 4096, 4096, 4096, 1, 0, 64, 512, b.SPECDEC_BF16,
                                  1.0, 0, b.SPECDEC_SAMPLE, 4096, 4096, None)
    assert rc == b.SPECDEC_ERR_UNSUPPORTED


@pytest.mark.gpu
@pytest.mark.parametrize("name,mode", [("llama3_8b_head", b.SPECDEC_SAMPLE),
                                       ("llama3_8b_head", b.SPECDEC_GREEDY),
                                       ("tiny_fp32", b.SPECDEC_SAMPLE)])
def test_noalloc_matches_workspace_entry_point(name, mode):
    import target_model_verify_gb300 as tv
    from target_model_verify_gb300 import build
    build.build()
    w = wl.get(name)
    assert b.specdec_verify_workspace_size(w.B, w.gamma, w.d, w.V,
                                           0 if w.dtype == "bf16" else 1, mode) <= SCRATCH_BYTES
    inp = wl.generate(w, 31, device="cuda:0")
    dl = inp["draft_logits"] if mode == b.SPECDEC_SAMPLE else None
    for call, seed in enumerate((1234, 98765)):          # two calls in a row
        ref_out, ref_nacc = tv.verify(inp["hidden"], inp["W_lm"], inp["draft_tokens"], dl,
                                      w.temperature, seed, mode)
        out = torch.full_like(ref_out, -7)
        nacc = torch.full_like(ref_nacc, -7)
        rc = _noalloc(inp, w.temperature, seed, mode, out, nacc, dl)
        assert rc == b.SPECDEC_OK, b.status_string(rc)
        torch.cuda.synchronize()
        # same kernels, same inputs and seed: the tokens agree exactly
        np.testing.assert_array_equal(out.cpu().numpy(), ref_out.cpu().numpy())
        np.testing.assert_array_equal(nacc.cpu().numpy(), ref_nacc.cpu().numpy())
        assert 0 <= int(nacc[0]) <= w.gamma


@pytest.mark.gpu
def test_noalloc_leftovers_of_other_shapes_and_a_failed_call_do_no_harm():
    """The shared array keeps whatever the previous call left: its header,
    fix-up tickets and sampler counters laid out for another shape or mode,
    or the state of a call that failed on the device. A sequence of calls
    of different shapes and modes, with one failed call in the middle (a
    draft token outside [0, V): that sequence reports n_accepted = -1 and
    -1 tokens), must give every valid call exactly the workspace entry
    point's tokens."""
    import target_model_verify_gb300 as tv
    from target_model_verify_gb300 import build
    build.build()
    llama = wl.get("llama3_8b_head", B=2)
    tiny = wl.get("tiny_fp32")
    x_llama = wl.generate(llama, 41, device="cuda:0")
    x_tiny = wl.generate(tiny, 42, device="cuda:0")
    bad = dict(x_llama, draft_tokens=x_llama["draft_tokens"].clone())
    bad["draft_tokens"][1, 2] = llama.V

    def check(w, inp, mode, seed):
        dl = inp["draft_logits"] if mode == b.SPECDEC_SAMPLE else None
        ref_out, ref_nacc = tv.verify(inp["hidden"], inp["W_lm"], inp["draft_tokens"], dl,
                                      w.temperature, seed, mode)
        out = torch.full_like(ref_out, -7)
        nacc = torch.full_like(ref_nacc, -7)
        assert _noalloc(inp, w.temperature, seed, mode, out, nacc, dl) == b.SPECDEC_OK
        torch.cuda.synchronize()
        np.testing.assert_array_equal(out.cpu().numpy(), ref_out.cpu().numpy())
        np.testing.assert_array_equal(nacc.cpu().numpy(), ref_nacc.cpu().numpy())

    check(llama, x_llama, b.SPECDEC_SAMPLE, 5)
    check(tiny, x_tiny, b.SPECDEC_SAMPLE, 6)
    check(llama, x_llama, b.SPECDEC_GREEDY, 7)
    out = torch.full((llama.B, llama.gamma + 1), -7, dtype=torch.int32, device="cuda:0")
    nacc = torch.full((llama.B,), -7, dtype=torch.int32, device="cuda:0")
    assert _noalloc(bad, 1.0, 8, b.SPECDEC_SAMPLE, out, nacc, bad["draft_logits"]) == b.SPECDEC_OK
    torch.cuda.synchronize()
    assert int(nacc[1]) == -1 and bool((out[1] == -1).all())
    assert 0 <= int(nacc[0]) <= llama.gamma
    check(llama, x_llama, b.SPECDEC_SAMPLE, 9)
    check(tiny, x_tiny, b.SPECDEC_SAMPLE, 10)
