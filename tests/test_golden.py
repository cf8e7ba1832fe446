"""Hand-worked examples with exact values (tests/golden/worked_examples.txt: the update rule
and closed form of page es, "Metodologia", items 2-3, evaluated by hand on inputs that make
every alpha a dyadic rational), met by the oracle (CPU) and by the CUDA paths (GPU: the
examples zero-padded to the supported widths)."""
import os

import numpy as np
import pytest

import oracle

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden", "worked_examples.txt")


def _examples():
    ex, cur = {}, None
    with open(GOLDEN) as f:
        for raw in f:
            line = raw.split("#", 1)[0].strip()
            if not line:
                continue
            if line.startswith("example "):
                _, name, dk, dv = line.split()
                cur = ex[name] = {"dk": int(dk), "dv": int(dv), "tokens": [], "o": [], "S": []}
            elif line.startswith("token "):
                k, v, beta, q = (p.split() for p in line[len("token "):].split("|"))
                cur["tokens"].append(([float(x) for x in k], [float(x) for x in v], float(beta[0]),
                                      [float(x) for x in q]))
            elif line.startswith("o "):
                cur["o"].append([float(x) for x in line.split(":", 1)[1].split()])
            elif line.startswith("S:"):
                cur["S"].append([float(x) for x in line.split(":", 1)[1].split()])
    return ex


EXAMPLES = _examples()


@pytest.mark.parametrize("name", sorted(EXAMPLES))
def test_oracle_meets_worked_example(name):
    e = EXAMPLES[name]
    L = len(e["tokens"])
    k = np.array([t[0] for t in e["tokens"]]).reshape(1, 1, L, e["dk"])
    v = np.array([t[1] for t in e["tokens"]]).reshape(1, 1, L, e["dv"])
    beta = np.array([t[2] for t in e["tokens"]]).reshape(1, 1, L)
    q = np.array([t[3] for t in e["tokens"]]).reshape(1, 1, L, e["dk"])
    o, S = oracle.fwd(q, k, v, beta)
    np.testing.assert_allclose(o[0, 0], np.array(e["o"]), rtol=0, atol=1e-14)
    np.testing.assert_allclose(S[0, 0], np.array(e["S"]), rtol=0, atol=1e-14)
    # the decode step applies the same update one token at a time
    St = np.zeros((1, 1, e["dk"], e["dv"]))
    for t in range(L):
        ot, St = oracle.step(q[:, :, t], k[:, :, t], v[:, :, t], beta[:, :, t], St)
        np.testing.assert_allclose(ot[0, 0], np.array(e["o"][t]), rtol=0, atol=1e-14)
    np.testing.assert_allclose(St[0, 0], np.array(e["S"]), rtol=0, atol=1e-14)


def test_fixture_betas_are_the_stated_logarithms():
    """The 17-digit beta literals are ln 2, ln(2)/4, ln 4 and ln(2)/2."""
    lits = {t[2] for e in EXAMPLES.values() for t in e["tokens"]}
    for want in (np.log(2), np.log(2) / 4, np.log(4), np.log(2) / 2):
        assert any(abs(b - want) <= 1e-16 for b in lits), want


def _padded(e, d, dtype, device):
    """The example's tokens zero-padded to width d (the extra key and value dimensions stay
    zero through the update, so the exact values carry over), as [1, 1, L, d] tensors."""
    import torch
    L = len(e["tokens"])
    q = torch.zeros((1, 1, L, d), dtype=torch.float64)
    k = torch.zeros_like(q)
    v = torch.zeros_like(q)
    beta = torch.zeros((1, 1, L), dtype=torch.float32)
    for t, (kt, vt, bt, qt) in enumerate(e["tokens"]):
        k[0, 0, t, :e["dk"]] = torch.tensor(kt)
        q[0, 0, t, :e["dk"]] = torch.tensor(qt)
        v[0, 0, t, :e["dv"]] = torch.tensor(vt)
        beta[0, 0, t] = bt
    return [x.to(dtype).to(device) for x in (q, k, v)] + [beta.to(device)]


@pytest.mark.gpu
@pytest.mark.parametrize("name", sorted(EXAMPLES))
@pytest.mark.parametrize("d,dtype,path,chunk,tol", [
    (16, "float32", "SIMT", 16, 1e-5),      # CUDA-core forward and decode step, fp32 inputs
    (128, "bfloat16", "TENSOR", 64, 1e-3),  # tcgen05 forward (fp16 operands), staged decode step
])
def test_cuda_path_meets_worked_example(name, d, dtype, path, chunk, tol):
    import torch
    import exact_flow_recurrence_gb300 as efla
    e = EXAMPLES[name]
    q, k, v, beta = _padded(e, d, getattr(torch, dtype), "cuda")
    o, S = efla.efla_fwd(q, k, v, beta, None, chunk=chunk, out_dtype=torch.float32, path=getattr(efla, path))
    efla.efla_get_status()
    o_want = torch.zeros((len(e["tokens"]), d), dtype=torch.float64)
    o_want[:, :e["dv"]] = torch.tensor(e["o"])
    S_want = torch.zeros((d, d), dtype=torch.float64)
    S_want[:e["dk"], :e["dv"]] = torch.tensor(e["S"])
    assert (o[0, 0].double().cpu() - o_want).abs().max().item() <= tol
    assert (S[0, 0].double().cpu() - S_want).abs().max().item() <= tol
    St = torch.zeros((1, 1, d, d), dtype=torch.float32, device="cuda")
    for t in range(len(e["tokens"])):
        qt, kt, vt, bt = (x[:, :, t].clone() for x in (q, k, v, beta))   # (16-byte aligned copies)
        ot = efla.efla_step(qt, kt, vt, bt, St, out_dtype=torch.float32)
        assert (ot[0, 0].double().cpu() - o_want[t]).abs().max().item() <= tol
    efla.efla_get_status()
    assert (St[0, 0].double().cpu() - S_want).abs().max().item() <= tol
