"""Kernels launched back to back on one stream that read each other's results.

Every library kernel is launched as a programmatic dependent of the kernel before
it on the stream: it may start while that kernel drains and waits for it to
finish before its first global-memory access.  These tests queue chains of GEMMs
with no host synchronisation in between, each stage's A being the previous
stage's C, then check every stage against the oracle applied to the input that
stage actually read (the previous stage's final output).  A stage that read its
input early would disagree with the oracle.  A chain is also captured into a CUDA
graph and replayed."""

import numpy as np
import pytest
import torch

import oracle
import synthetic
from oracle import compare

import dense_matrix_multiply_gb300 as g

pytestmark = pytest.mark.gpu

SEED = 31  # seed block of these problems


@pytest.fixture(scope="module", autouse=True)
def _lib(lib):
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    return lib


def band_rows(M):
    rows = set()
    for b0 in range(0, M, 256):
        for off in (0, 37, 70, 101, 133, 168, 200, 255):
            if b0 + off < M:
                rows.add(b0 + off)
    return np.array(sorted(rows), dtype=np.int64)


def host_bits(t, dtype):
    h = t.cpu().numpy()
    return h if dtype == "f32" else h.view(np.uint16)


def dev(buf):
    return torch.from_numpy(buf if buf.dtype == np.float32 else buf.view(np.int16)).cuda()


def queue_chain(dtype, M, dims, seed):
    """Device input X [M, dims[0]] and, for each stage s, weights [dims[s], dims[s+1]]
    (normal, scaled by 1/sqrt(K) so values stay O(1)) and an output buffer."""
    tdt = torch.float32 if dtype == "f32" else torch.int16
    x = synthetic.matrix(dtype, M, dims[0], seed, "normal", 1.0)
    ws = [synthetic.matrix(dtype, dims[s], dims[s + 1], seed + 1 + s, "normal", 1.0 / np.sqrt(dims[s]))
          for s in range(len(dims) - 1)]
    dx = dev(x)
    dws = [dev(w) for w in ws]
    outs = [torch.full((M * dims[s + 1],), -1, dtype=tdt, device="cuda") for s in range(len(dims) - 1)]
    return x, ws, dx, dws, outs


def run_chain(dtype, M, dims, dx, dws, outs):
    fn = {"f32": g.gemm_f32_rm, "bf16": g.gemm_bf16_rm}[dtype]
    a = dx
    kernels = []
    for s in range(len(dims) - 1):
        fn(a, dws[s], outs[s], M, dims[s + 1], dims[s])
        kernels.append(g.gemm_last_kernel())
        a = outs[s]
    return kernels


def check_chain(dtype, M, dims, x, ws, outs):
    variant = dtype + "_rm"
    a = x
    rows = np.arange(M) if M <= 64 else band_rows(M)
    for s in range(len(dims) - 1):
        K, N = dims[s], dims[s + 1]
        c = host_bits(outs[s], dtype)
        ref, S = oracle.gemm_rows(variant, a, ws[s], M, N, K, rows)
        got = (c.astype(np.float64) if dtype == "f32" else
               (c.astype(np.uint32) << 16).view(np.float32).astype(np.float64)).reshape(M, N)[rows]
        res = compare.check(variant, got, ref, S, K)
        assert res["ok"], (s, res)
        a = c  # the next stage read exactly this


CHAINS = [
    ("bf16", 8, [1024, 4096, 2048, 12288, 1024], "skinny kernel (strips alone and on clusters)"),
    ("bf16", 1, [4096, 4096, 12288, 1024], "skinny kernel at M = 1"),
    ("bf16", 8, [1024, 20480, 4096, 20480, 512], "256-column skinny kernel (160 strips) between 128-column ones"),
    ("bf16", 1, [4100, 4096, 1024], "GEMV (X rows of 8200 bytes), then the skinny kernel"),
    ("bf16", 2048, [3072, 2560, 3072, 2560], "CTA pairs, stream-K tail on the 2560-wide stages"),
    ("bf16", 512, [1024, 2048, 520, 1024], "CTA pairs, ragged N then ragged K"),
    ("f32", 256, [512, 1024, 256, 768], "packed-FMA SIMT kernel"),
    ("f32", 4, [1024, 3000, 1024], "FP32 GEMV"),
    ("f32", 2304, [1024, 1664, 2432], "packed-FMA SIMT kernel, last round split into half-K CTA pairs"),
]


@pytest.mark.parametrize("case", CHAINS, ids=lambda c: f"{c[0]}-M{c[1]}-{'x'.join(map(str, c[2]))}")
def test_back_to_back_chain(case):
    dtype, M, dims, _what = case
    x, ws, dx, dws, outs = queue_chain(dtype, M, dims, synthetic.seed_for(SEED, 0) + 100 * CHAINS.index(case))
    run_chain(dtype, M, dims, dx, dws, outs)  # no synchronisation between the stages
    g.gemm_synchronize()
    torch.cuda.synchronize()
    check_chain(dtype, M, dims, x, ws, outs)


def test_chain_captured_in_a_cuda_graph():
    """The same chains captured into one CUDA graph (stream-ordered scratch of the
    stream-K tail becomes graph memory nodes; the SGEMM's split last round a
    programmatic edge to a cluster launch) and replayed twice: the results equal
    the eager ones bit for bit."""
    cases = [CHAINS[0], CHAINS[2], CHAINS[4], CHAINS[6], CHAINS[8]]
    eager, staged = [], []
    for case in cases:
        dtype, M, dims, _ = case
        x, ws, dx, dws, outs = queue_chain(dtype, M, dims, synthetic.seed_for(SEED, 1) + 100 * cases.index(case))
        run_chain(dtype, M, dims, dx, dws, outs)
        g.gemm_synchronize()
        torch.cuda.synchronize()
        eager.append([o.clone() for o in outs])
        staged.append((dtype, M, dims, dx, dws, outs))
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        for dtype, M, dims, dx, dws, outs in staged:
            run_chain(dtype, M, dims, dx, dws, outs)
    for _ in range(2):
        for _, _, _, _, _, outs in staged:
            for o in outs:
                o.fill_(-1)
        graph.replay()
        torch.cuda.synchronize()
        g.gemm_synchronize()
        for want, (_, _, _, _, _, outs) in zip(eager, staged):
            for w, o in zip(want, outs):
                assert torch.equal(w, o)
