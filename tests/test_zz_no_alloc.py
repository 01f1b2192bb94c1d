"""The decode entry point for callers that cannot allocate device memory.

`mla_decode_static_scratch` runs the same decode as `mla_decode` but keeps its split
plan and partial results in a fixed scratch array owned by the library, instead of a
workspace the caller allocates.  This file checks it through the C ABI against the
ordinary entry point on two calls in a row (the second call finds the first call's
leftovers in the shared array), and that requests too large for the array are refused.
It lives in a file of its own, collected last.
"""
import ctypes

import pytest
import torch

import mla_latent_kv_77_b300 as mla
from mla_latent_kv_77_b300 import workloads
from helpers import check_lse, check_out, oracle_decode

pytestmark = pytest.mark.gpu


def _static_call(q, pool, bt, sl, case, num_splits, o_lat, lse):
    vp = lambda t: ctypes.c_void_p(t.data_ptr())
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    return mla.lib().mla_decode_static_scratch(vp(q), vp(pool), vp(bt), vp(sl), case.B, case.Tq, 128,
                                               pool.shape[0], bt.shape[1], float(case.scale),
                                               int(case.causal), num_splits, vp(o_lat), vp(lse), stream)


def test_static_scratch_matches_workspace_entry_point_two_calls_in_a_row():
    calls = [
        # first call: forced splits, so partial results pass through the scratch array
        dict(seq_lens=[64 * 13 + 7, 64 * 5, 90], shuffle=True, seed=31, splits=3, Tq=1, causal=False),
        # second call: different queries, lengths and plan, on top of the first call's leftovers
        dict(seq_lens=[64 * 9 + 1, 260], shuffle=True, seed=32, splits=0, Tq=2, causal=True),
    ]
    for c in calls:
        case = workloads.make_case("static", c["seq_lens"], Tq=c["Tq"], causal=c["causal"], shuffle=c["shuffle"],
                                   seed=c["seed"])
        q, pool = case.q_abs.cuda(), case.pool.cuda()
        bt, sl = case.block_table.cuda(), case.seq_lens.cuda()
        ref_o, ref_l = mla.decode(q, pool, bt, sl, case.scale, causal=case.causal, num_splits=c["splits"])
        o = torch.empty_like(ref_o)
        l = torch.empty_like(ref_l)
        assert _static_call(q, pool, bt, sl, case, c["splits"], o, l) == mla.Status.OK
        torch.cuda.synchronize()
        assert mla.get_device_status() == (0, 0)
        # same plan, same inputs, deterministic kernels: the results must be bit-identical, so
        # that leftovers of the previous call in the shared array cannot hide under a tolerance
        assert torch.equal(o.view(torch.int16), ref_o.view(torch.int16))
        assert torch.equal(l.view(torch.int32), ref_l.view(torch.int32))
        check_out(o, ref_o.double().cpu().numpy(), "o_lat (static scratch)")
        check_lse(l, ref_l.double().cpu().numpy())
        # and against the fp64 oracle directly
        or_o, or_l = oracle_decode(case)
        check_out(o, or_o, "o_lat (static scratch) vs oracle")
        check_lse(l, or_l)


def test_static_scratch_refuses_requests_larger_than_the_array():
    case = workloads.make_case("static_big", [64], seed=33)
    q, pool = case.q_abs.cuda(), case.pool.cuda()
    bt, sl = case.block_table.cuda(), case.seq_lens.cuda()
    o = torch.empty(case.B, 1, 128, 512, dtype=torch.bfloat16, device="cuda")
    l = torch.empty(case.B, 1, 128, dtype=torch.float32, device="cuda")
    # the smallest batch whose workspace exceeds the array (91 queries with the automatic
    # plan; 90 is the largest admitted) is refused before anything runs
    limit = 64 << 20  # MLA_STATIC_SCRATCH_BYTES
    n_big = 1
    while mla.decode_workspace_size(n_big, 1, 0) <= limit:
        n_big += 1
    assert mla.decode_workspace_size(n_big - 1, 1, 0) <= limit < mla.decode_workspace_size(n_big, 1, 0)
    big = workloads.make_case("static_big", [64] * n_big, seed=34)
    st = _static_call(big.q_abs.cuda(), big.pool.cuda(), big.block_table.cuda(), big.seq_lens.cuda(), big, 0,
                      torch.empty(n_big, 1, 128, 512, dtype=torch.bfloat16, device="cuda"),
                      torch.empty(n_big, 1, 128, dtype=torch.float32, device="cuda"))
    assert st == mla.Status.WORKSPACE
    # forced splits push a small batch over the limit too
    assert _static_call(q, pool, bt, sl, case, 4000, o, l) == mla.Status.WORKSPACE
    # and a request within the limit still works afterwards
    assert _static_call(q, pool, bt, sl, case, 0, o, l) == mla.Status.OK
    ref_o, ref_l = mla.decode(q, pool, bt, sl, case.scale)
    torch.cuda.synchronize()
    check_out(o, ref_o.double().cpu().numpy())
    check_lse(l, ref_l.double().cpu().numpy())
