"""The entry points keep the planner's recent plans in a small per-thread table. Whatever the order
of the queries, and whether the table holds a plan or has to make it again, every (shape, options)
query must get the plan the planner makes for it: checked against a fresh thread (an empty table)
over more distinct queries than the table holds, including one shape under several options."""
import threading

import pytest

pytestmark = pytest.mark.gpu

QUERIES = [
    (8, 2112, 7168, 0, 0, 0), (8, 2112, 7168, 3, 4, 0), (8, 2112, 7168, 1, 0, 0), (8, 2112, 7168, 2, 2, 0),
    (8, 2112, 7168, 2, 0, 32), (16, 3072, 1536, 0, 0, 0), (16, 3072, 1536, 3, 2, 0), (32, 4096, 512, 0, 0, 0),
    (32, 4096, 512, 3, 0, 32), (64, 7168, 2048, 0, 0, 0), (64, 7168, 2048, 2, 2, 0), (256, 4096, 7168, 0, 0, 0),
    (256, 3072, 1536, 0, 0, 0), (256, 3072, 1536, 2, 0, 128), (4, 2880, 512, 0, 0, 0), (32, 2880, 512, 0, 0, 0),
    (16, 2112, 7168, 0, 0, 0), (1, 128, 65536, 0, 0, 0), (100, 300, 512, 0, 0, 0), (129, 256, 2048, 0, 0, 0),
    (513, 2048, 1024, 0, 0, 0), (2048, 4096, 7168, 0, 0, 0), (24, 2112, 7168, 0, 0, 0), (5, 200, 520, 0, 0, 0),
]


def _plans(order):
    import block_scaled_mxfp4_bf16_gb300 as mx
    return {q: mx.mxfp4_gemm_plan(*q) for q in order}


def test_cached_plans_equal_fresh_plans():
    import torch
    torch.cuda.set_device(0)
    fresh = {}

    def worker():
        torch.cuda.set_device(0)
        fresh.update(_plans(QUERIES))

    t = threading.Thread(target=worker)
    t.start()
    t.join()
    assert len(fresh) == len(QUERIES)
    # this thread: forwards, backwards and interleaved, three times the table's size in queries
    for order in (QUERIES, QUERIES[::-1], QUERIES[::2] + QUERIES[1::2]):
        got = _plans(order)
        for q in QUERIES:
            assert got[q] == fresh[q], q
    # the same shape under different options gets different plans (the options are in the key)
    assert fresh[(8, 2112, 7168, 1, 0, 0)]["path"] == 1 and fresh[(8, 2112, 7168, 0, 0, 0)]["path"] == 3
    assert fresh[(8, 2112, 7168, 3, 4, 0)]["splits"] == 4
    assert fresh[(8, 2112, 7168, 2, 0, 32)]["m_tile"] == 16       # a 32-token request cut to M rounded up to 16
    assert fresh[(256, 3072, 1536, 2, 0, 128)]["m_tile"] == 128 and fresh[(256, 3072, 1536, 0, 0, 0)]["m_tile"] == 64
