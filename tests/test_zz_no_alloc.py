"""The static-scratch entry point (spec_verify_static) called through the C ABI: it must give the same
results as spec_verify with a caller workspace, on two calls in a row. Kept in its own file, collected last,
so that it runs both after the rest of the GPU suite and alone in a fresh process."""
import ctypes

import numpy as np
import pytest
import torch

import oracle
import speculative_decoding_verification_target_gb300 as sv
import workloads
from parity_util import assert_chain, assert_diag, host

pytestmark = pytest.mark.gpu


def _p(t):
    return ctypes.c_void_p(t.data_ptr() if t is not None else 0)


def _static_call(lib, inp, w, stream):
    B, K, V = w.B, w.K, w.V
    dev = inp["target"].device
    acc = torch.full((B,), -7, dtype=torch.int32, device=dev)
    out = torch.full((B, K + 1), -7, dtype=torch.int32, device=dev)
    diag = torch.zeros((B, K, 4), dtype=torch.float32, device=dev)
    status = ctypes.c_uint32(0xFFFFFFFF)
    dtype = 0 if inp["target"].dtype == torch.bfloat16 else 1
    rc = lib.spec_verify_static(_p(inp["target"]), _p(inp["draft"]), dtype, _p(inp["tokens"]), _p(inp["seeds"]), B,
                                K, V, ctypes.c_float(w.temperature), _p(acc), _p(out), _p(diag),
                                ctypes.byref(status), ctypes.c_void_p(stream.cuda_stream))
    assert rc == 0, lib.spec_last_error()
    return acc, out, diag, status.value


@pytest.mark.parametrize("name,B", [("sps_llama3_b64_k5", 16), ("tiny_sps_v1000", 8)])
def test_static_scratch_matches_workspace_entry(name, B):
    lib = sv.load()
    lib.spec_debug_set_stats_grid(0)
    w = workloads.WORKLOADS[name].scaled(B=B)
    stream = torch.cuda.current_stream()
    for call in range(2):   # two calls in a row: the second reuses the region the first one left behind
        inp = workloads.make(w.scaled(gen_seed=w.gen_seed + 31 * call), device="cuda")
        ref = sv.verify(inp["target"], inp["draft"], inp["tokens"], inp["seeds"], w.temperature)
        acc, out, diag, status = _static_call(lib, inp, w, stream)
        torch.cuda.synchronize()
        assert status == 0
        assert torch.equal(acc, ref["accept_len"])
        assert torch.equal(out, ref["out_tokens"])
        assert np.abs(diag.cpu().numpy() - ref["diag"].cpu().numpy()).max() <= 1e-6
        assert sv.read_status(ref["workspace"]) == 0


def test_static_scratch_reports_bad_tokens_per_call():
    lib = sv.load()
    w = workloads.WORKLOADS["tiny_sps_v1000"].scaled(B=4)
    inp = workloads.make(w, device="cuda")
    stream = torch.cuda.current_stream()
    bad = dict(inp)
    bad["tokens"] = inp["tokens"].clone()
    bad["tokens"][1, 2] = w.V + 5
    _, _, _, status = _static_call(lib, bad, w, stream)
    assert status == 1   # SPEC_STATUS_BAD_TOKEN for this call
    _, _, _, status = _static_call(lib, inp, w, stream)
    assert status == 0   # cleared by the next call


def test_static_scratch_against_the_oracle():
    """The static-scratch call checked directly against the fp64 oracle: an fp32 workload whose V is not a
    multiple of 8 (rows not 16-byte aligned: element-wise loads), then a bf16 one, back to back."""
    lib = sv.load()
    stream = torch.cuda.current_stream()
    for w in (workloads.WORKLOADS["tiny_sps_v1000"].scaled(B=6, V=1001),
              workloads.WORKLOADS["sps_llama3_b64_k5"].scaled(B=8, gen_seed=77)):
        inp = workloads.make(w, device="cuda")
        ref = oracle.verify(host(inp["target"]), host(inp["draft"]), inp["tokens"].cpu().numpy(),
                            inp["seeds"].cpu().numpy().astype(np.uint64), w.temperature)
        acc, out, diag, status = _static_call(lib, inp, w, stream)
        torch.cuda.synchronize()
        assert status == 0
        got = {"accept_len": acc, "out_tokens": out, "diag": diag}
        assert_diag(got, ref)
        assert_chain(got, ref, w.K)
