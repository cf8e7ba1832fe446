"""Failure detection without a GPU fault: a bounded device-side wait that nothing will
satisfy gives up, records EFLA_ERR_TIMEOUT in the library's status word, and leaves the
context usable (the same bounded-wait helpers guard every tensor-core kernel)."""
import ctypes

import pytest
import torch

import efla_workloads as wl
import exact_flow_recurrence_gb300 as efla
from parity import TOL_BF16, assert_close
import oracle

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("kind", [0, 1])   # 0: mbarrier never completed, 1: flag never set
def test_bounded_wait_reports_timeout_and_context_survives(kind):
    efla.efla_get_status()                      # start from a clear status word
    efla.efla_wait_selftest(kind, limit=2048)
    with pytest.raises(efla.EflaError) as ei:
        efla.efla_get_status()
    assert ei.value.status == 6                 # EFLA_ERR_TIMEOUT
    efla.efla_get_status()                      # the word was cleared by the read
    # the context still runs the forward correctly
    w = wl.resized(wl.LM340M_FWD, B=1, H=2, L=70)
    x = wl.make_inputs(w)
    d = {n: (t.cuda() if t is not None else None) for n, t in x.items()}
    o, Sf = efla.efla_fwd(d["q"], d["k"], d["v"], d["beta"], d["S0"], chunk=w.chunk)
    efla.efla_get_status()
    o_ref, _ = oracle.fwd(x["q"][:, :1], x["k"][:, :1], x["v"][:, :1], x["beta"][:, :1], None)
    assert_close("o[0,0]", o[:, :1], o_ref, TOL_BF16, stored_bf16=True)


def test_wait_selftest_rejects_bad_arguments():
    lib = efla.load_library()
    assert lib.efla_wait_selftest(2, 10, None) == 1
    assert lib.efla_wait_selftest(0, 0, None) == 1
