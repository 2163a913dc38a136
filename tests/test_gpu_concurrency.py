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


@pytest.mark.parametrize("names", [("swiglu", "downproj"), ("backward", "fp8")])
def test_two_threads_two_streams(names):
    shapes = {"swiglu": (1024, 2048, 512), "downproj": (768, 1024, 640), "backward": (768, 1536, 512),
              "fp8": (1024, 1024, 512)}
    jobs = [_setup(n, *shapes[n]) for n in names]
    refs = []
    for w, inp, plan, out in jobs:  # each alone, first
        _run(plan, inp, out)
        torch.cuda.synchronize()
        refs.append((out.C.clone(), None if out.row_out is None else out.row_out.clone(),
                     None if out.col_out is None else out.col_out.clone(),
                     None if out.C8 is None else out.C8.clone(), None if out.amax is None else out.amax.item()))
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
    for (w, inp, plan, out), (c_ref, r_ref, col_ref, c8_ref, amax_ref) in zip(jobs, refs):
        assert plan.query_status(out.workspace) == 0
        assert torch.equal(out.C, c_ref), "%s: C differs from the run alone" % w.name
        if c8_ref is not None:
            assert torch.equal(out.C8, c8_ref), "%s: C8 differs from the run alone" % w.name
        if amax_ref is not None:
            assert out.amax.item() == amax_ref  # a maximum does not depend on the order
        if r_ref is not None:
            np.testing.assert_allclose(out.row_out.cpu().numpy(), r_ref.cpu().numpy(), rtol=RED_TOL)
        if col_ref is not None:
            c = out.C.double()
            bound = RED_TOL * c.abs().sum(0) + 1e-6
            assert torch.all((out.col_out.double() - col_ref.double()).abs() <= bound)
