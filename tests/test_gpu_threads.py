"""Several host threads calling the library at once, each on its own stream with its own buffers:
the per-thread plan table, the kernels' one-time attribute set-up (first calls racing), the
per-stream default workspaces and prepared calls must give every thread the same bits a single
thread gets. The shapes cover the weight-resident, fused, two-kernel and wide-tile plans, so
first calls of different kernels race too."""
import threading

import pytest
import torch

from block_scaled_mxfp4_bf16_gb300 import workloads

pytestmark = pytest.mark.gpu

SHAPES = [(8, 2112, 7168, 0), (5, 300, 520, 1), (64, 1024, 2048, 2), (300, 384, 1536, 2), (16, 3072, 1536, 0)]


def test_concurrent_threads_match_one_thread():
    import block_scaled_mxfp4_bf16_gb300 as mx
    torch.cuda.set_device(0)
    cases = []
    for i, (M, N, K, path) in enumerate(SHAPES):
        bq, bs = mx.mxfp4_quantize(workloads.random_bf16(N, K, seed=300 + i).cuda())
        packed = mx.mxfp4_prepack_b(bq, bs)
        a = workloads.random_bf16(M, K, seed=400 + i).cuda()
        cases.append((M, N, K, path, a, packed))
    torch.cuda.synchronize()
    want = [mx.mxfp4_gemm(a, packed, N, path=path) for (M, N, K, path, a, packed) in cases]
    torch.cuda.synchronize()

    results, errors = {}, []
    start = threading.Barrier(len(cases) * 2)

    def worker(t):
        try:
            torch.cuda.set_device(0)
            M, N, K, path, a, packed = cases[t % len(cases)]
            stream = torch.cuda.Stream()
            c = torch.empty(M, N, dtype=torch.bfloat16, device="cuda")
            with torch.cuda.stream(stream):
                start.wait()
                for i in range(20):
                    if i % 2:
                        mx.mxfp4_gemm(a, packed, N, c=c, path=path, stream=stream)
                    else:
                        mx.prepare_gemm(a, packed, N, c, path=path, stream=stream)()
            stream.synchronize()
            results[t] = c
        except Exception as e:   # reported below, on the main thread
            errors.append((t, repr(e)))

    threads = [threading.Thread(target=worker, args=(t,)) for t in range(len(cases) * 2)]
    for th in threads:
        th.start()
    for th in threads:
        th.join(timeout=120)
    assert not errors, errors
    assert len(results) == len(threads)
    for t, c in results.items():
        w = want[t % len(cases)]
        assert torch.equal(c.view(torch.int16), w.view(torch.int16)), (t, SHAPES[t % len(cases)])
    assert mx.mxfp4_device_status() == 0
