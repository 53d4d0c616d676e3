"""The Python binding's own argument checks, which run before any library
call: host (CPU) tensors and wrong dtypes are refused with ValueError, so no
device pointer is ever formed from host memory.  No GPU is needed."""
import numpy as np
import pytest
import torch

import nvfp4_quantization_gb300 as nq


def cpu_plan(E=4, T=8, k=2):
    z = lambda n: torch.zeros(n, dtype=torch.int32)
    return nq.RoutePlan(z(E + 1), z(E), z(T * k), T, k, E, 128, 1024, torch.zeros(1, dtype=torch.int32))


def test_host_tensors_are_refused():
    tok = torch.zeros((8, 512), dtype=torch.bfloat16)
    topk = torch.zeros((8, 2), dtype=torch.int32)
    with pytest.raises(ValueError, match="CUDA"):
        nq.ep_route_plan(topk, 4)
    with pytest.raises(ValueError, match="CUDA"):
        nq.ep_nvfp4_pack(tok, cpu_plan())
    with pytest.raises(ValueError, match="CUDA"):
        nq.ep_nvfp4_dispatch(tok, topk, 4)
    with pytest.raises(ValueError, match="CUDA"):
        nq.ep_nvfp4_direct_receive(torch.zeros((128, 304), dtype=torch.uint8), 512, torch.zeros(5, dtype=torch.int32), 4)


def test_wrong_dtypes_are_refused_before_the_device_check():
    # the dtype is checked together with the device; a host tensor of the
    # wrong dtype still fails the device check first, with ValueError
    with pytest.raises(ValueError):
        nq.ep_route_plan(torch.zeros((8, 2), dtype=torch.int64), 4)
    with pytest.raises(ValueError):
        nq.ep_nvfp4_pack(torch.zeros((8, 512), dtype=torch.float32), cpu_plan())


def test_row_bytes_and_capacity_match_the_header_formulas():
    for H in (16, 256, 1024, 1056, 4096, 7168, 16384):
        assert nq.row_bytes(H) == (9 * H // 16 + 16 + 15) // 16 * 16
    # the header's bound on R = sum_e ceil(c_e / A) * A: T*k + E*(A-1)
    for T, k, E, A in ((8, 2, 4, 128), (4096, 2, 16, 128), (700, 1, 3, 256), (0, 2, 4, 128)):
        assert nq.rows_capacity(T, k, E, A) == T * k + E * (A - 1)
    # and it is an upper bound: brute force over every way 5 slots fall into 3 experts
    import itertools
    for counts in itertools.product(range(6), repeat=3):
        if sum(counts) == 5:
            R = sum(-(-c // 128) * 128 for c in counts)
            assert R <= nq.rows_capacity(5, 1, 3, 128)
