"""Large sums and cumulative sums on several streams at once.

Each stream has its own page of control words (tickets, chunk queue, digit
accumulators, fallback flags), which every call leaves zero.  Calls that
take different paths (the double sum's first and second pass, its
Inf/NaN pass, the general float kernel, the cumulative sums' fast and
general paths) run concurrently on four streams and must each give the
oracle's bits."""
import numpy as np
import pytest
import torch

import oracle
from compensated_bit_reproducible_gb300 import api, inputs
from tests.gpu_util import dev, same_bits, to_dev

pytestmark = pytest.mark.gpu
F32, F64 = np.float32, np.float64


def test_concurrent_streams():
    dev()
    n = 300_003
    m = 150_001                      # cumulative sums: above the fast-path threshold
    wide = inputs.wide_f64(n, seed=31)
    outl = wide.copy()
    outl[n // 2] = -4.0e240          # above the sampled bins: second pass
    nan = inputs.inject_specials(wide, "nan", seed=32)
    flt = inputs.normal_f32(n, seed=33)
    cs = inputs.wide_f64(m, seed=34)
    asc = np.sort(np.abs(cs)) * np.sign(cs)   # the index settles late: general path
    sums = [wide, outl, nan, flt]
    want_sum = [np.array([oracle.adn_sum(x, 3, "fp")], x.dtype)[0] for x in sums]
    want_cs = [oracle.adn_cumsum(x, 3) for x in (cs, asc)]
    d_sums = [to_dev(x) for x in sums]
    d_cs = [to_dev(x) for x in (cs, asc)]
    streams = [torch.cuda.Stream() for _ in range(4)]
    reps = 6
    outs = {}
    torch.cuda.synchronize()
    for r in range(reps):
        for k, s in enumerate(streams):
            with torch.cuda.stream(s):
                # every stream runs every kind of call, in a different order
                for j in range(len(sums)):
                    i = (j + k) % len(sums)
                    o = torch.empty(1, dtype=d_sums[i].dtype, device=d_sums[i].device)
                    api.repro_sum_async(d_sums[i], o, 3, stream=s)
                    outs[("sum", r, k, i)] = o
                for i in ((k + r) % 2, (k + r + 1) % 2):
                    outs[("cs", r, k, i)] = api.repro_cumsum(d_cs[i], K=3, stream=s)
    torch.cuda.synchronize()
    for key, o in outs.items():
        kind, r, k, i = key
        got = o.cpu().numpy()
        if kind == "sum":
            want = want_sum[i]
            if np.isnan(want):
                assert np.isnan(got[0]), key
            else:
                assert same_bits(got[0], want), key
        else:
            assert same_bits(got, want_cs[i]), key
