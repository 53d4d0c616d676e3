"""GPU parity over a seeded sweep of random shapes: the whole path (route plan
and pack in one dispatch call with the per-expert amax reduced by the pack,
direct receive in the linear or the tiled scale layout, unpack, MXFP8 pack)
against the oracle, byte for byte.  Each case draws its own token count, hidden
size (a multiple of 32, ragged against the kernels' 64-, 256- and 512-column
units), expert count, top-k, dropped slots, rounding mode and token scales, the
latter spread over many binades in some cases so that 16-row blocks whose token
exponents differ by more than 13 (the receive's FP32 decode-table fallback)
occur alongside all-zero tokens."""
import numpy as np
import pytest

import workloads
from paths import DeviceRun, OracleRun, compare_runs

pytestmark = pytest.mark.gpu

N_CASES = 12


def random_workload(case: int) -> workloads.Workload:
    rng = np.random.default_rng(9100 + case)
    T = int(rng.integers(1, 1500))
    # odd cases: a multiple of 512 (the pack's warp-per-token kernel); even: any multiple of 32
    H = 512 * int(rng.integers(1, 4)) if case % 2 else 32 * int(rng.integers(1, 41))
    E = int(rng.integers(1, 81))
    k = int(rng.integers(1, min(8, E) + 1))
    x = rng.standard_normal((T, H)).astype(np.float32)
    spread = int(rng.choice([0, 4, 40]))   # binades of the per-token scale
    x *= np.exp2(rng.integers(-spread, spread + 1, size=(T, 1))).astype(np.float32)
    x[rng.random(T) < 0.02] = 0.0          # whole tokens of zeros
    topk = np.argsort(rng.random((T, E)), axis=1)[:, :k].astype(np.int32)
    topk[rng.random((T, k)) < float(rng.choice([0.0, 0.05, 0.3]))] = -1
    rounding = int(rng.integers(0, 2))
    return workloads.Workload(name=f"sweep{case}", description="random shape", tokens=workloads.to_bf16_bits(x),
                              topk=topk, E=E, rounding=rounding, seed=int(rng.integers(0, 1 << 31)))


@pytest.mark.parametrize("case", range(N_CASES))
def test_random_shapes(case):
    w = random_workload(case)
    swz = w.H % 128 == 0 and case % 4 < 2
    g = DeviceRun(w, unpack=True, mxfp8=True, dispatch=True, amax=True, swizzled=swz)
    o = OracleRun(w, g.R_cap, unpack=True, mxfp8=True)
    compare_runs(g, o)
