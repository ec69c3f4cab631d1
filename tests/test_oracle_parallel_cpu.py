"""The threaded oracle helpers the full-size GPU tests use must return
exactly what single calls of the oracle return: splitting an extend request
into pieces of new tokens (piece t0..t1 = an extend over C + t0 cached
tokens) and dealing decode requests to threads change no value."""
import numpy as np
import torch

import oracle
import workloads
from tests import gpu_util as gu


def test_parallel_extend_equals_one_call():
    case = workloads.make_extend_case("par", num_q_heads=4, num_kv_heads=2, head_dim=64,
                                      num_reqs=3, prefix_len=37, ext_lo=5, ext_hi=90, budget=4096,
                                      seed=11)
    pool_t, per_batch = workloads.make_extend_values(case, "cpu")
    hk, hv = gu.u16(pool_t[0, 0]), gu.u16(pool_t[1, 0])
    b = case.batches[0]
    k, v, q = per_batch[0]
    orc = oracle.get()
    orc.store_kv(hk, hv, k, v, b.out_loc)
    ref = orc.extend(q, hk, hv, b.page_table, b.cached_lens, b.extend_lens, case.sm_scale)
    got = gu.parallel_oracle_extend(hk, hv, q, b.page_table, b.cached_lens, b.extend_lens,
                                    b.q_offsets, case.sm_scale, chunk=7)
    assert np.array_equal(got, ref)


def test_parallel_decode_equals_one_call():
    case = workloads.decode_tiny()
    pool_t, k_new, v_new, q = workloads.make_decode_values(case, "cpu")
    hk, hv = gu.u16(pool_t[0, 0]), gu.u16(pool_t[1, 0])
    orc = oracle.get()
    ref, ref_lse = orc.decode(q[0], hk, hv, case.page_table, case.seq_lens, case.sm_scale)
    got, lse = gu.parallel_oracle_decode(hk, hv, q[0], case.page_table, case.seq_lens, case.sm_scale)
    assert np.array_equal(got, ref) and np.array_equal(lse, ref_lse)
    sub = [3, 1]
    got2, _ = gu.parallel_oracle_decode(hk, hv, q[0], case.page_table, case.seq_lens, case.sm_scale,
                                        reqs=sub)
    assert np.array_equal(got2, ref[sub])
