"""Failure detection on the GPU without a fault: a bounded device-side wait that runs out is
reported through the workspace status word, and the CUDA context stays usable (GPU)."""
import numpy as np
import pytest
import torch

from state_space_model_scan_gb300 import _lib
from state_space_model_scan_gb300 import inputs as I
from helpers import TOL, rel_l2, gpu_forward, oracle_forward, flat

pytestmark = pytest.mark.gpu


def test_bounded_wait_expiry_is_reported_and_the_context_survives():
    ws = torch.zeros(4096, dtype=torch.uint8, device="cuda")
    assert _lib.selftest_bounded_wait(ws, 50) == _lib.SSD_OK
    assert _lib.query_status(ws) == 6          # SSD_ERR_DEVICE_TIMEOUT: nobody set the flag
    # the same context still runs the scan correctly afterwards
    w = I.Workload("t", 1, 300, 4, 64, 2, 128, 128, "bf16", has_z=True, has_init=True)
    inp = I.make_inputs(w)
    y, fin = gpu_forward(w, inp, algo="fused")
    yo, fo = oracle_forward(w, inp)
    assert rel_l2(flat(y, 300), yo) <= TOL["bf16"]
    assert rel_l2(fin.double().cpu().numpy(), fo) <= TOL["bf16"]


def test_bounded_wait_arguments():
    ws = torch.zeros(4096, dtype=torch.uint8, device="cuda")
    assert _lib.selftest_bounded_wait(ws, 0) == 1
    assert _lib.selftest_bounded_wait(ws, 2001) == 1
    assert _lib.selftest_bounded_wait(ws[:64], 10) == 1
