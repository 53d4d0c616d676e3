"""ep_route_plan_noalloc, the routing entry point that allocates nothing.

It exists for callers that cannot allocate device memory for a workspace (a
runtime that owns the whole GPU's memory in its own pool, a loop where a
cudaMalloc would stall the device): it keeps its scratch in a fixed array
inside the library instead.  Its plan must be identical, byte for byte, to the
oracle's plan and to ep_route_plan's on the same inputs -- routing is integer
work -- including on consecutive calls, where the scratch still holds the
previous call's totals and barrier words.

The file is named so that pytest collects it last: a run that stops at the
first failure has run every other test before this one.  Outputs are
allocated by the test (torch); the entry point itself is called through the
C ABI with raw pointers.
"""
import ctypes

import numpy as np
import pytest
import torch

import nvfp4_quantization_gb300 as nq
import oracle
from nvfp4_quantization_gb300 import _lib

pytestmark = pytest.mark.gpu


def _topk(T, E, k, seed):
    rng = np.random.default_rng(seed)
    topk = np.argsort(rng.random((T, E)), axis=1)[:, :k].astype(np.int32)
    topk[rng.random((T, k)) < 0.02] = -1
    return torch.from_numpy(topk).cuda()


def _p(t):
    return ctypes.c_void_p(t.data_ptr())


def _noalloc_plan(topk, E, A=128):
    """Outputs allocated here, then one call of the C entry point."""
    T, k = topk.shape
    R_cap = nq.rows_capacity(T, k, E, A)
    dev = topk.device
    off = torch.full((E + 1,), -7, dtype=torch.int32, device=dev)
    cnt = torch.full((E,), -7, dtype=torch.int32, device=dev)
    dest = torch.full((max(T * k, 1),), -7, dtype=torch.int32, device=dev)
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    s = _lib.lib().ep_route_plan_noalloc(_p(topk), T, k, E, A, R_cap, _p(off), _p(cnt), _p(dest), _p(st),
                                         ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert s == 0, _lib.status_string(s)
    return off, cnt, dest, st


def _same_plan(topk, E, got):
    """The no-alloc plan equals the oracle's plan of the same routing (the
    definition), and ep_route_plan's (the library's other entry point)."""
    ref = nq.ep_route_plan(topk, E, 128)
    torch.cuda.synchronize()
    off, cnt, dest, st = got
    T, k = topk.shape
    o_off, o_cnt, o_dest, o_st = oracle.route_plan(topk.cpu().numpy(), E, 128)
    assert np.array_equal(off.cpu().numpy(), o_off)
    assert np.array_equal(cnt.cpu().numpy(), o_cnt)
    assert np.array_equal(dest[: T * k].cpu().numpy(), o_dest[: T * k])
    assert int(st.item()) == int(o_st) == 0
    assert torch.equal(off.cpu(), ref.offsets.cpu())
    assert torch.equal(cnt.cpu(), ref.counts.cpu())
    assert torch.equal(dest[: T * k].cpu(), ref.dest[: T * k].cpu())
    assert int(ref.status.item()) == 0


# (T, E, k): the register fast path at the 16K-token, 256-expert top-8 size;
# k > 8 (general kernel); more 512-token chunks than resident CTAs (several
# chunks per CTA); a tiny case; T = 0.
SHAPES = [(16384, 256, 8), (3000, 32, 12), (400000, 64, 2), (37, 8, 2), (0, 4, 2)]


@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "x".join(map(str, s)))
def test_two_calls_in_a_row_match_ep_route_plan(shape):
    T, E, k = shape
    a = _topk(T, E, k, seed=T + E)
    b = _topk(T, E, k, seed=T + E + 1)
    got_a = _noalloc_plan(a, E)
    got_b = _noalloc_plan(b, E)      # same scratch, straight after the first call
    torch.cuda.synchronize()
    _same_plan(a, E, got_a)
    _same_plan(b, E, got_b)


def test_large_then_small_then_large():
    """A smaller problem after a larger one (stale totals beyond its own
    rows), then the larger one again."""
    big, small = _topk(16384, 256, 8, seed=1), _topk(700, 16, 2, seed=2)
    r1 = _noalloc_plan(big, 256)
    r2 = _noalloc_plan(small, 16)
    r3 = _noalloc_plan(big, 256)
    torch.cuda.synchronize()
    _same_plan(big, 256, r1)
    _same_plan(small, 16, r2)
    _same_plan(big, 256, r3)


def test_rejects_a_problem_larger_than_the_scratch():
    E, k = 256, 2
    T = (_lib.EP_ROUTE_STATIC_SCRATCH_BYTES // (E * 4) + 1) * 512      # one chunk too many
    assert nq.lib().ep_route_workspace_bytes(T, k, E) > _lib.EP_ROUTE_STATIC_SCRATCH_BYTES
    fake = ctypes.c_void_p(0x10000)    # never reached: the size check comes first
    s = _lib.lib().ep_route_plan_noalloc(fake, T, k, E, 128, nq.rows_capacity(T, k, E, 128), fake, fake, fake,
                                         fake, None)
    assert s == -4      # EP_ERR_CAPACITY
