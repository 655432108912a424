"""The process pool the full-size parity tests use returns the same errors as
the oracle called directly (CPU only)."""

import numpy as np
import torch

import workloads
from oracle import ns as ons
from oracle_pool import OraclePool, bf16_bits_to_f64


def _bits(t):
    return t.contiguous().view(torch.int16).numpy().view(np.uint16).reshape(-1)


def test_bf16_bits_decode_exactly():
    t = workloads.gen_tensor((7, 9), 1.0, 11, 0)
    assert np.array_equal(bf16_bits_to_f64(_bits(t)).reshape(7, 9), t.double().numpy())


def test_pool_errors_equal_direct_oracle():
    shapes = [(12, 20), (20, 12), (4, 3, 5)]
    jobs, want = [], {}
    for i, s in enumerate(shapes):
        t = workloads.gen_tensor(s, 1.0, 12, i)
        y = (t.float() * 0.5 + 0.01).to(torch.bfloat16)          # a stand-in "result"
        y32 = t.float() * 0.75
        ref = ons.newton_schulz(t.double().numpy(), 3, 3.4445, -4.775, 2.0315, 1e-7)
        want[("bf16", i)] = ons.rel_fro_error(y.double().numpy(), ref)
        want[("f32", i)] = ons.rel_fro_error(y32.double().numpy(), ref)
        jobs.append((("bf16", i), s, _bits(t), _bits(y), 3, 3.4445, -4.775, 2.0315, 1e-7, 0.0))
        jobs.append((("f32", i), s, _bits(t), y32.numpy().reshape(-1).view(np.uint32), 3, 3.4445, -4.775,
                     2.0315, 1e-7, 0.0))
    with OraclePool(workers=2) as pool:
        got = pool.errors(jobs)
    assert got.keys() == want.keys()
    for k in want:
        # single- and multi-threaded BLAS may round the products differently
        assert abs(got[k] - want[k]) <= 1e-12 * max(1.0, want[k]), k
