"""psattn_decode_noalloc: the decode entry point for callers that cannot
allocate device memory (a process whose HBM is already owned by another
allocator, such as an engine that reserves almost all of it for its KV-cache
pool, or a latency-critical path where cudaMalloc/cudaFree, which can
synchronise the device, are not allowed).  Its workspace lives in a fixed
array inside the library instead of a per-plan cudaMalloc.

Checked through the C ABI against psattn_decode on two calls in a row, and
for the clear rejection of a plan whose workspace does not fit.  This file is
collected last so that a run that stops at the first failure has already run
every other test; it also passes on its own in a fresh process.
"""
import numpy as np
import pytest

import workloads as W

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


def test_noalloc_matches_decode_two_calls():
    import oracle
    import shared_prefix_kv_gb300 as ps
    from workloads.device import DeviceProblem, shape_of, tolerances

    p = W.make("llama8b", small=True)
    o_ref, l_ref = oracle.attention(p)
    d = DeviceProblem(p)
    with d.plan() as pl:
        d.decode(pl)
        ref_out, ref_lse = d.result()
        assert pl.status() == (0, 0)
    t_out, t_lse = tolerances(p)
    sms = torch.cuda.get_device_properties(torch.cuda.current_device()).multi_processor_count
    with ps.Plan(shape_of(p), p.block_table, p.group_of_req, p.group_parent, p.prefix_len,
                 p.suffix_len, host_only_sms=sms) as hp:
        stream = torch.cuda.current_stream().cuda_stream
        for _ in range(2):
            d.out.fill_(float("nan"))
            d.lse.fill_(float("nan"))
            ps.psattn_decode_noalloc(hp.handle, d.q, d.pool, d.bt, d.gor, d.plen, d.slen, d.out,
                                     d.lse, stream)
            out, lse = d.result()
            assert np.isfinite(out).all() and np.isfinite(lse).all()
            assert np.abs(out - ref_out).max() <= t_out
            assert np.abs(lse - ref_lse).max() <= t_lse
            assert np.abs(out - o_ref).max() <= t_out
            assert np.abs(lse - l_ref).max() <= t_lse


def test_noalloc_ragged_chunked_batch():
    """A batch with prefill chunks in the ragged form (per-row limits read
    from the plan's request table) through the no-allocation entry point."""
    import dataclasses

    import oracle
    import shared_prefix_kv_gb300 as ps
    from shared_prefix_kv_gb300 import chunked
    from workloads.device import DeviceProblem, shape_of, tolerances

    p, ql, q = W.make_chunked(seed=7, small=True)
    sh, bt, gor, gpar, plen, slen, leaf = chunked.expand_ragged(
        shape_of(p), p.block_table, p.group_of_req, p.group_parent, p.prefix_len, p.suffix_len, ql)
    p2 = dataclasses.replace(p, q=q, block_table=bt, group_of_req=gor, group_parent=gpar,
                             prefix_len=plen, suffix_len=slen)
    d = DeviceProblem(p2)
    sms = torch.cuda.get_device_properties(torch.cuda.current_device()).multi_processor_count
    with ps.Plan(shape_of(p2), bt, gor, gpar, plen, slen, host_only_sms=sms, leaf_len=leaf) as hp:
        ps.psattn_decode_noalloc(hp.handle, d.q, d.pool, d.bt, d.gor, d.plen, d.slen, d.out,
                                 d.lse, torch.cuda.current_stream().cuda_stream)
        out, lse = d.result()
    o_ref, l_ref = oracle.attention_chunked(p, ql, q)
    t_out, t_lse = tolerances(p)
    assert np.isfinite(out).all() and np.isfinite(lse).all()
    assert np.abs(out - o_ref).max() <= t_out
    assert np.abs(lse - l_ref).max() <= t_lse


def test_noalloc_rejects_plan_beyond_scratch():
    import shared_prefix_kv_gb300 as ps

    # 8192 ungrouped requests of 4000 tokens: about 134 MB of partial slots,
    # more than the fixed scratch array holds.  Rejected before any launch, so
    # the device pointers below are never read.
    R, S, B = 8192, 4000, 16
    nb = -(-S // B)
    bt = np.arange(R * nb, dtype=np.int32).reshape(R, nb)
    sh = ps.make_shape(R, 0, 32, 8, 128, B, nb, R * nb, ps.BF16, 128 ** -0.5)
    with ps.Plan(sh, bt, np.full(R, -1, np.int32), None, None, np.full(R, S, np.int32),
                 host_only_sms=152) as hp:
        x = torch.zeros(64, device="cuda", dtype=torch.bfloat16)
        lse = torch.zeros(64, device="cuda")
        with pytest.raises(ps.PsattnError) as e:
            ps.psattn_decode_noalloc(hp.handle, x, x, x, x, x, x, x, lse, 0)
        assert e.value.status == ps.ERR_NOMEM
