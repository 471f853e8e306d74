"""pod_run_static_scratch: POD for callers that cannot allocate device memory.

Such callers (a plugin whose host application owns every device allocation, a
process under a fixed device-memory budget, a serving loop that cannot take
cudaMalloc's implicit synchronisation) get the kernels' scratch from a fixed
array inside the library instead of a workspace of their own. These tests go
through the C ABI (ctypes binding) and check that this entry point returns
what pod_run returns with a caller-allocated workspace, on calls in a row
that use different plans (one under RoPE, whose angle table and rotated
copies also live in the array and must be rebuilt when another plan used it
in between, and one with a custom prefill mask, whose bits live there too),
and that a plan too large for the array is refused. The file
name sorts after every other test file on purpose: a run that stops at the
first failure has run all the others before this one.
"""
import numpy as np
import pytest
import torch

import prefill_decode_paged_pod_gb300 as pod
from pod_workloads import make_config, make_custom, with_prefill_custom_mask
from podtest_util import LSE_ATOL, OUT_ATOL, OUT_RTOL, to_dev


@pytest.fixture(scope="module", autouse=True)
def built():
    from prefill_decode_paged_pod_gb300 import _build
    _build.build()
    pod.load_library()


def _close(ref, got):
    ref = ref.double().cpu().numpy()
    got = got.double().cpu().numpy()
    assert np.all(np.isfinite(got))
    return np.all(np.abs(got - ref) <= OUT_ATOL + OUT_RTOL * np.abs(ref))


def test_static_scratch_refuses_oversized_plan():
    # one decode request over 10M single-token pages: the page table alone
    # needs 40 MB of metadata, more than the 32 MiB array
    n = 10_000_000
    h = pod.pod_plan(None, None, None, None,
                     np.array([0, 1]), np.array([0, n]), np.arange(n, dtype=np.int32),
                     np.array([1]), 8, 1, 64, 1, True, -1, None, dtype=torch.float16,
                     p_num_pages=1, d_num_pages=n, num_sms=8)
    assert pod.pod_workspace_size(h) > pod.pod_static_scratch_capacity()
    with pytest.raises(pod.PodError) as e:
        pod.pod_run_static_scratch(h, None, None, None, None)
    assert e.value.code == 3 and "static scratch" in str(e.value)


@pytest.mark.gpu
def test_static_scratch_matches_pod_run_two_calls():
    cases = [
        # split decode KV (partials and the merge kernel live in the scratch)
        make_custom("split", torch.bfloat16, 16, 2, 128, 16, True, -1, [40], [300],
                    [1, 2, 1], [5000, 7000, 3000], seed=11, sinks=True),
        make_config("c1"),
        make_custom("rope", torch.bfloat16, 16, 2, 128, 16, True, -1, [70], [100], [1, 4],
                    [300, 129], seed=13),
        make_config("c1"),
        with_prefill_custom_mask(
            make_custom("mask", torch.float16, 8, 2, 64, 16, False, -1, [90, 40], [200, 40],
                        [1, 1], [100, 33], seed=15), seed=16, density=0.5),
        make_config("c1"),
    ]
    cases[2].rope = (1.0, 1e4)
    sms = [4, 0, 0, 0, 0, 0]
    for inp, ns in zip(cases, sms):
        dev = to_dev(inp)
        # existing entry point, caller-allocated workspace
        h_ref = pod.plan_inputs(inp, workspace=None, num_sms=ns)
        ws = torch.empty(pod.pod_workspace_size(h_ref), dtype=torch.uint8, device="cuda")
        pod.pod_bind_workspace(h_ref, ws)
        ref = pod.pod_run(h_ref, dev["q_p"], dev["kv_p"], dev["q_d"], dev["kv_d"], ws,
                          sinks=dev["sinks"])
        # the no-allocation entry point, on a host-only plan of the same inputs
        h = pod.plan_inputs(inp, workspace=None, num_sms=ns)
        got = pod.pod_run_static_scratch(h, dev["q_p"], dev["kv_p"], dev["q_d"], dev["kv_d"],
                                         sinks=dev["sinks"])
        torch.cuda.synchronize()
        for name, r, g in zip(("out_p", "lse_p", "out_d", "lse_d"), ref, got):
            if r.numel() == 0:
                continue
            if name.startswith("lse"):
                # rows a custom mask leaves without keys have lse = -inf on both
                assert torch.equal(torch.isinf(r), torch.isinf(g)), name
                fin = torch.isfinite(r)
                assert float((r[fin] - g[fin]).abs().max()) <= LSE_ATOL, name
            else:
                assert _close(r, g), name
        pod.pod_destroy(h)
        pod.pod_destroy(h_ref)
