"""linrec_scan_f32_host: the scan on host buffers with pipelined copies, against the oracle."""
import numpy as np
import pytest
import torch

import linear_recurrence_scan_fp32_gb300 as lr
import oracle
from linear_recurrence_scan_fp32_gb300 import inputs
from tests._util import assert_close

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda:0")


@pytest.fixture(scope="module", autouse=True)
def _built():
    from linear_recurrence_scan_fp32_gb300 import _build
    _build.build()
    torch.cuda.set_device(DEV)


@pytest.mark.parametrize("name", ["pages", "long", "tiny"])
def test_host_pipeline_workloads(name):
    w = inputs.WORKLOADS[name]
    a, b = inputs.generate_workload(w)
    h64, _ = oracle.f64(a, b)
    a_p, b_p = a.pin_memory(), b.pin_memory()
    del a, b
    s = torch.cuda.Stream()
    h = lr.linrec_scan_f32_host(a_p, b_p, stream=s)
    s.synchronize()
    assert_close(h.numpy(), h64, f"{name} through the host pipeline")
    # a second call into the same output, on the default stream
    h.fill_(float("nan"))
    lr.linrec_scan_f32_host(a_p, b_p, h)
    torch.cuda.synchronize()
    assert_close(h.numpy(), h64, f"{name} second call")


@pytest.mark.parametrize("shape", [(3, 1000, 260), (1, 3_000_000, 4), (5, 7, 33), (2, 1, 8)],
                         ids=lambda s: "x".join(map(str, s)))
def test_host_pipeline_shapes_and_pageable_memory(shape):
    B, L, D = shape
    a, b = inputs.generate(B, L, D, seed=70 + L, a_dist="u[0.5,1)", b_dist="n(0,1)")
    h64, _ = oracle.f64(a, b)
    h = torch.empty_like(a)                         # pageable
    lr.linrec_scan_f32_host(a, b, h)
    torch.cuda.synchronize()
    assert_close(h.numpy(), h64, f"{shape} pageable")


def test_host_pipeline_refuses_overlap_and_device_tensors():
    a = torch.zeros(1, 10, 4)
    with pytest.raises(lr.LinrecError) as e:
        lr.linrec_scan_f32_host(a, a, a)
    assert e.value.code == lr.LINREC_ERR_ALIAS
    with pytest.raises(TypeError):
        lr.linrec_scan_f32_host(a.to(DEV), a.to(DEV))


def test_host_pipeline_mixed_memory_takes_the_copy_path():
    """Pinned inputs with a pageable output: the pieces go through the copy pipeline."""
    w = inputs.WORKLOADS["pages"]
    a, b = inputs.generate_workload(w)
    h64, _ = oracle.f64(a, b)
    h = torch.empty_like(a)                         # pageable
    lr.linrec_scan_f32_host(a.pin_memory(), b.pin_memory(), h)
    torch.cuda.synchronize()
    assert_close(h.numpy(), h64, "pinned in, pageable out")
