"""Concurrent use of the C ABI (needs a GB300): two host threads, each with
its own plan, outputs, workspace and CUDA stream, launch repeatedly at the
same time.  The library keeps no per-run host state outside the plan and
the caller's workspace (its error string is per thread), so every output
must equal the same plan's output run alone: bit for bit where the program
has no atomics, within the reduction tolerance where it does."""
import threading

import numpy as np
import pytest
import torch

from gemm_epilogue_transformer_smem_gb300 import api, synth

from parity import RED_TOL

pytestmark = pytest.mark.gpu

DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def _lib(cuda_lib):
    return cuda_lib


def _setup(name, M, N, K):
    w = synth.WORKLOADS[name].scaled(M, N, K)
    inp = synth.make_inputs(w, DEV)
    plan = api.Plan(w.M, w.N, w.K, w.program, b_layout=w.b_layout)
    out = api.allocate_outputs(plan, DEV)
    return w, inp, plan, out


def _run(plan, inp, out):
    api.run_program(plan, inp.A, inp.B, out, alpha=inp.alpha, fp8_scale=inp.fp8_scale, bias=inp.bias, aux=inp.aux)


def test_two_threads_two_streams():
    jobs = [_setup("swiglu", 1024, 2048, 512), _setup("downproj", 768, 1024, 640)]
    refs = []
    for w, inp, plan, out in jobs:  # each alone, first
        _run(plan, inp, out)
        torch.cuda.synchronize()
        refs.append((out.C.clone(), None if out.row_out is None else out.row_out.clone()))
        out.C.fill_(0)
    errors = []

    def worker(job):
        w, inp, plan, out = job
        try:
            s = torch.cuda.Stream()
            with torch.cuda.stream(s):
                for _ in range(25):
                    _run(plan, inp, out)
            s.synchronize()
        except Exception as e:  # surfaced below
            errors.append(e)

    threads = [threading.Thread(target=worker, args=(j,)) for j in jobs]
    for t in threads:
        t.start()
    for t in threads:
        t.join(timeout=120)
    assert not errors, errors
    for (w, inp, plan, out), (c_ref, r_ref) in zip(jobs, refs):
        assert plan.query_status(out.workspace) == 0
        assert torch.equal(out.C, c_ref), "%s: C differs from the run alone" % w.name
        if r_ref is not None:
            np.testing.assert_allclose(out.row_out.cpu().numpy(), r_ref.cpu().numpy(), rtol=RED_TOL)
