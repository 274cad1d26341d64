"""The all-gather + GEMM from pinned host shards (kosmos_ag_gemm_host): the
shard copies (into x_gathered) and output copies run on two copy streams and
overlap the kernel through per-shard arrival words and output-tile counts per
group of tile rows; the kernel copies each shard on into its device buffer.
Results must equal kosmos_ag_gemm on the same shards bit for bit (every
schedule, both tile engines, full size), x_gathered and the device shard
buffers must hold the shards; a failed kernel releases the output waits so
that no stream blocks, and the status reports the failure."""
import numpy as np
import pytest
import torch

from _helpers import bf16_tensor_to_f64, kosmos, rel_err
from kosmos_inputs import WORKLOADS, ag_inputs, bf16_bits, sample_indices

pytestmark = pytest.mark.gpu
TOL = 1e-2


@pytest.fixture(scope="module")
def K():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    return kosmos()


def run_host(K, inp, o=None, reps=1):
    P = len(inp["x"])
    m, k = inp["x"][0].shape
    n = inp["w"].shape[1]
    hx = [x.pin_memory() for x in inp["x"]]
    xd = [torch.empty(m, k, dtype=torch.bfloat16, device="cuda") for _ in range(P)]
    w = inp["w"].cuda()
    xg = torch.empty(P * m, k, dtype=torch.bfloat16, device="cuda")
    yd = torch.empty(P * m, n, dtype=torch.bfloat16, device="cuda")
    hy = torch.empty(P * m, n, dtype=torch.bfloat16).pin_memory()
    ws = K.workspace(K.OP_AG_GEMM, P, m, n, k, o=o)
    h2d, d2h = torch.cuda.Stream(), torch.cuda.Stream()
    outs = []
    for _ in range(reps):
        hy.fill_(float("nan"))
        K.ag_gemm_host(hx, xd, w, xg, yd, hy, ws, o, h2d_stream=h2d, d2h_stream=d2h)
        torch.cuda.current_stream().synchronize()
        outs.append(hy.clone())
    return outs, ws, xg, xd


def run_dev(K, inp, o=None):
    P = len(inp["x"])
    m, k = inp["x"][0].shape
    n = inp["w"].shape[1]
    xs = [x.cuda() for x in inp["x"]]
    w = inp["w"].cuda()
    xg = torch.empty(P * m, k, dtype=torch.bfloat16, device="cuda")
    y = torch.empty(P * m, n, dtype=torch.bfloat16, device="cuda")
    ws = K.workspace(K.OP_AG_GEMM, P, m, n, k, o=o)
    K.ag_gemm(xs, w, xg, y, ws, o)
    K.check(ws)
    return y.cpu()


@pytest.mark.parametrize("shape", [(4, 384, 256, 768), (3, 200, 192, 264), (2, 1, 64, 8)])  # whole, ragged, one row
@pytest.mark.parametrize("pair", [1, 0])
@pytest.mark.parametrize("sched", [0, 1, 2])
def test_ag_host_small_matches_device_call(K, orc, sched, pair, shape):
    P, m, k, n = shape
    inp = ag_inputs(P, m, k, n, seed=41, var_w=1.0 / k)
    o = K.opts(sched=sched, cta_pair=pair)
    outs, ws, xg, xd = run_host(K, inp, o, reps=2)
    K.check(ws, "ag_gemm_host")
    assert torch.equal(outs[0], outs[1])
    assert torch.equal(outs[0], run_dev(K, inp, o))
    assert torch.equal(xg.cpu(), torch.cat(inp["x"], 0))
    for r in range(P):
        assert torch.equal(xd[r].cpu(), inp["x"][r]), f"device shard buffer {r}"
    ref = orc.ag_gemm([bf16_bits(x) for x in inp["x"]], bf16_bits(inp["w"]))
    assert rel_err(bf16_tensor_to_f64(outs[0]), ref) <= TOL


def test_ag_host_full_size(K, orc):
    w = WORKLOADS["ag_bf16_p8"]
    inp = ag_inputs(w.P, w.m, w.k, w.n, w.seed, w.var_x, w.var_w)
    outs, ws, xg, xd = run_host(K, inp, reps=2)
    K.check(ws, "ag_gemm_host")
    assert torch.equal(outs[0], outs[1])
    assert torch.equal(outs[0], run_dev(K, inp))
    assert torch.equal(xg.cpu(), torch.cat(inp["x"], 0))
    for r in range(w.P):
        assert torch.equal(xd[r].cpu(), inp["x"][r]), f"device shard buffer {r}"
    rows = np.unique(np.concatenate([sample_indices(w.P * w.m, 8, seed=3), np.arange(w.P) * w.m]))
    ref = orc.ag_gemm([bf16_bits(x) for x in inp["x"]], bf16_bits(inp["w"]), rows=rows)
    assert rel_err(bf16_tensor_to_f64(outs[0][torch.from_numpy(rows)]), ref) <= TOL


@pytest.mark.parametrize("pair", [1, 0])
def test_ag_host_failed_kernel_releases_output_waits(K, pair):
    """A shard copied to the device whose arrival word is never written: the
    kernel times out, its output waits are released, every stream completes
    and the status says TIMEOUT; after a workspace re-init the next call is
    correct."""
    P, m, k, n = 2, 128, 128, 256
    inp = ag_inputs(P, m, k, n, seed=9, var_w=1.0 / k)
    o = K.opts(inject=K.INJECT_DROP_ARRIVAL | (1 << 32), wait_limit_ns=2_000_000, cta_pair=pair)
    outs, ws, _, _ = run_host(K, inp, o)
    st, ent = K.status_sync(ws)
    assert st == K.ERR_TIMEOUT, f"status {st}, entry {ent}"
    K.workspace_init(ws)
    torch.cuda.synchronize()
    hx = [x.pin_memory() for x in inp["x"]]
    xd = [torch.empty(m, k, dtype=torch.bfloat16, device="cuda") for _ in range(P)]
    wd = inp["w"].cuda()
    xg = torch.empty(P * m, k, dtype=torch.bfloat16, device="cuda")
    yd = torch.empty(P * m, n, dtype=torch.bfloat16, device="cuda")
    hy = torch.empty(P * m, n, dtype=torch.bfloat16).pin_memory()
    K.ag_gemm_host(hx, xd, wd, xg, yd, hy, ws, K.opts(cta_pair=pair), h2d_stream=torch.cuda.Stream(),
                   d2h_stream=torch.cuda.Stream())
    torch.cuda.synchronize()
    K.check(ws)
    assert torch.equal(hy, run_dev(K, inp))
