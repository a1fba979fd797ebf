"""Thread safety of shared handles: host threads call the library's entry
points that run library GEMMs (mdcn_backward on two workloads and the
ablation mdcn_forward_im2col_gemm) at the same time, each on its own stream
with its own workspace, several times, while a fourth thread runs the fused
forward. Every result must equal the one the same call gives when nothing
else runs: bitwise for the forwards and for every gradient but grad_x, and
within the parity gate for grad_x, whose fp32 atomic sums may change order
from run to run.
"""
import threading

import pytest
import torch

import modulated_deformable_convolution_gb300 as mdcn
from modulated_deformable_convolution_gb300.workloads import CONFIGS, make_grad_out, make_inputs

pytestmark = pytest.mark.gpu

TOL = {"f32": 1e-4, "f16": 2e-2, "bf16": 2e-2}
REPEATS = 6


def _dev_inputs(case):
    dev = torch.device("cuda", 0)
    return {k: (None if v is None else v.to(dev)) for k, v in make_inputs(case).items()}


class BackwardJob:
    def __init__(self, h, case):
        self.case = case
        self.h = h
        self.d = _dev_inputs(case)
        self.go = make_grad_out(case).to(self.d["x"].device)
        d = self.d
        self.gb = torch.empty_like(d["bias"]) if d["bias"] is not None else None
        self.g = [torch.empty_like(d[k]) for k in ("x", "offset", "mask", "weight")]
        self.ws = torch.empty(mdcn.mdcn_backward_workspace_size(h, d["x"], d["offset"], d["mask"], d["weight"],
                                                                self.gb), dtype=torch.uint8, device=d["x"].device)

    def run(self, stream):
        d = self.d
        mdcn.mdcn_backward(self.h, d["x"], d["offset"], d["mask"], d["weight"], self.go, *self.g, self.gb, self.ws,
                           stream)

    def result(self):
        return [t.clone() for t in self.g] + ([self.gb.clone()] if self.gb is not None else [])


class AblationJob:
    def __init__(self, h, case):
        self.h = h
        self.d = d = _dev_inputs(case)
        self.out = torch.empty(mdcn.mdcn_output_dims(h, d["x"], d["offset"], d["mask"], d["weight"], d["bias"]),
                               dtype=d["x"].dtype, device=d["x"].device)
        self.ws = torch.empty(mdcn.mdcn_im2col_gemm_workspace_size(h, d["x"], d["offset"], d["mask"], d["weight"],
                                                                   d["bias"]), dtype=torch.uint8,
                              device=d["x"].device)

    def run(self, stream):
        d = self.d
        mdcn.mdcn_forward_im2col_gemm(self.h, d["x"], d["offset"], d["mask"], d["weight"], d["bias"], self.out,
                                      self.ws, stream)

    def result(self):
        return [self.out.clone()]


class FusedJob(AblationJob):
    def __init__(self, h, case):
        self.h = h
        self.d = d = _dev_inputs(case)
        self.out = torch.empty(mdcn.mdcn_output_dims(h, d["x"], d["offset"], d["mask"], d["weight"], d["bias"]),
                               dtype=d["x"].dtype, device=d["x"].device)
        self.ws = torch.empty(mdcn.mdcn_workspace_size(h, d["x"], d["offset"], d["mask"], d["weight"], d["bias"]),
                              dtype=torch.uint8, device=d["x"].device)

    def run(self, stream):
        d = self.d
        mdcn.mdcn_forward(self.h, d["x"], d["offset"], d["mask"], d["weight"], d["bias"], self.out, self.ws, stream)


def test_threads_on_one_handle_match_serial_results():
    # one handle shared by every thread (the header allows it); two workloads
    # with different GEMM shapes so that interleaved stream or workspace
    # settings would show
    a = CONFIGS["neck_f16"]
    b = CONFIGS["multidg_bf16"]
    h_a = mdcn.Handle(**a.attrs())
    h_b = mdcn.Handle(**b.attrs())
    jobs = [BackwardJob(h_a, a), AblationJob(h_b, b), BackwardJob(h_b, b), FusedJob(h_a, a)]
    streams = [torch.cuda.Stream() for _ in jobs]
    serial = []
    for job, st in zip(jobs, streams):
        with torch.cuda.stream(st):
            job.run(st)
            serial.append(job.result())
        st.synchronize()

    errors = []
    results = [[] for _ in jobs]
    start = threading.Barrier(len(jobs))

    def worker(i):
        try:
            torch.cuda.set_device(0)
            start.wait()
            for _ in range(REPEATS):
                with torch.cuda.stream(streams[i]):
                    jobs[i].run(streams[i])
                    results[i].append(jobs[i].result())  # copied on the job's stream, before its next run
                streams[i].synchronize()
        except Exception as e:  # reported below
            errors.append((i, repr(e)))

    threads = [threading.Thread(target=worker, args=(i,)) for i in range(len(jobs))]
    for t in threads:
        t.start()
    for t in threads:
        t.join()
    assert not errors, errors
    for i, job in enumerate(jobs):
        tol = TOL[job.d["x"].dtype == torch.float32 and "f32" or "f16"]
        for rep, res in enumerate(results[i]):
            for j, (got, ref) in enumerate(zip(res, serial[i])):
                label = f"job {i} ({type(job).__name__}) repeat {rep} tensor {j}"
                if isinstance(job, BackwardJob) and j == 0:
                    # grad_x: fp32 atomic sums, order may differ
                    scale = ref.float().abs().max().item()
                    err = (got.float() - ref.float()).abs().max().item()
                    assert err <= tol * scale, f"{label}: {err} > {tol} * {scale}"
                else:
                    assert torch.equal(got, ref), label
