"""GPU parity: libpkv (through its C ABI) against the CPU oracle.

Appends and block copies are compared bit for bit over the whole pool
(including the NaN-poisoned rows nobody wrote); attention outputs and LSEs
element by element within |gpu - ref| <= 2e-3 + 1e-2 |ref|.
"""
import numpy as np
import pytest
import torch

import oracle
from paged_kv_cache_41_gb300 import pkv
from paged_kv_cache_41_gb300 import workloads as wl

import parity_util as pu

pytestmark = pytest.mark.gpu


def _run_batch(b, partition_size=0, rows=None, check_pool=True):
    kc, vc = pu.device_pool(b)
    pu.device_fill(b, kc, vc)
    hk, hv = pu.host_pool(b)
    pu.oracle_fill(b, hk, hv)
    torch.cuda.synchronize()
    assert pkv.get_device_error() == 0
    if check_pool:
        assert pu.pools_equal_bytes(kc, hk), "K pool differs from the oracle's after kv_append"
        assert pu.pools_equal_bytes(vc, hv), "V pool differs from the oracle's after kv_append"
    out, lse = pu.device_decode(b, kc, vc, partition_size)
    assert pkv.get_device_error() == 0
    ref, ref_lse = pu.oracle_decode(b, hk, hv, rows)
    if rows is not None:
        out, lse = out[rows], lse[rows]
    pu.assert_close(out, ref, f"{b.name} out")
    pu.assert_close(lse, ref_lse, f"{b.name} lse")
    return kc, vc


def test_tiny_fp32_append_and_decode():
    b = wl.tiny_batch(device="cuda")
    _run_batch(b)


@pytest.mark.parametrize("partition_size", [16, 32, 48, 64])
def test_tiny_fp32_split_k(partition_size):
    b = wl.tiny_batch(device="cuda")
    _run_batch(b, partition_size=partition_size)


EDGE_LENS = [1, 15, 16, 17, 31, 32, 33, 100, 257, 0, 1000, 64, 2]


@pytest.mark.parametrize("dtype,d,hq,hkv,p", [
    ("bf16", 128, 32, 8, 16), ("bf16", 128, 8, 8, 16), ("bf16", 128, 16, 8, 16),
    ("bf16", 128, 64, 8, 16), ("bf16", 64, 8, 2, 16), ("f32", 128, 8, 2, 16),
    ("f32", 64, 4, 2, 16), ("bf16", 128, 32, 8, 64), ("bf16", 128, 32, 8, 32),
    ("bf16", 128, 32, 8, 128), ("bf16", 64, 16, 4, 256), ("f32", 128, 16, 2, 192),
    ("bf16", 128, 16, 4, 96),
    # eight query heads per kv head on the CUDA cores: fp32 pools, and bf16
    # at head_dim 64 (the tensor cores take bf16 at 128 only)
    ("f32", 128, 16, 2, 16), ("bf16", 64, 16, 2, 16), ("f32", 64, 16, 2, 32),
])
@pytest.mark.parametrize("partition_size", [0, "one_block", "three_blocks", "whole"])
def test_edge_lengths(dtype, d, hq, hkv, p, partition_size):
    b = wl.custom_batch(EDGE_LENS, dtype=dtype, hq=hq, hkv=hkv, d=d, p=p, seed=31, device="cuda")
    ps = {0: 0, "one_block": p, "three_blocks": 3 * p,
          "whole": b.max_blocks * p}[partition_size]
    _run_batch(b, partition_size=ps)


# Eight query heads per kv head run on the tensor cores (128-row stages);
# these cover every block size that path takes, ragged and empty lengths,
# pieces cut at every stage boundary, and the NaN-poisoned stale rows.
G8_LENS = [1, 127, 128, 129, 255, 0, 700, 16, 2000, 33]


@pytest.mark.parametrize("p", [16, 32, 64, 128, 256])
@pytest.mark.parametrize("partition_size", [0, 128, 384, "whole"])
def test_gqa8_tensor_core_decode(p, partition_size):
    b = wl.custom_batch(G8_LENS, dtype="bf16", hq=64, hkv=8, d=128, p=p, seed=61, device="cuda")
    ps = b.max_blocks * p if partition_size == "whole" else partition_size
    if ps % p:
        ps = p * ((ps + p - 1) // p)
    _run_batch(b, partition_size=ps)


@pytest.mark.parametrize("rep", range(3))
def test_gqa8_tensor_core_decode_one_stage_segments(rep):
    # every (sequence, kv head) segment fits one 128-row stage, so every stage
    # starts a new piece with its own Q: a CTA's first stages load three
    # pieces' Q back to back, before any of their MMAs need have run
    lens = np.random.default_rng(70 + rep).integers(1, 128, size=400, endpoint=True)
    b = wl.custom_batch(lens, dtype="bf16", hq=64, hkv=8, d=128, p=16, seed=70 + rep,
                        device="cuda")
    _run_batch(b, check_pool=False)


@pytest.mark.parametrize("hq,hkv,batch", [(32, 8, 2500), (64, 8, 1700)])
def test_batch_past_one_scan_pass(hq, hkv, batch):
    # more sequences than one pass of the CTAs' length scan covers (1024 for
    # the CUDA-core decode, 1536 for the tensor-core one): the multi-pass
    # search for each CTA's first stage
    lens = np.random.default_rng(batch).integers(0, 48, size=batch, endpoint=True)
    b = wl.custom_batch(lens, dtype="bf16", hq=hq, hkv=hkv, d=128, p=16, seed=batch, device="cuda")
    _run_batch(b, check_pool=False)


@pytest.mark.parametrize("d,p", [(64, 16), (128, 32)])
def test_short_segments_past_the_descriptor_batches(d, p):
    # more than 64 stages per CTA and a piece end at nearly every stage: the
    # consumers read the next stage's descriptor (its q) at each piece end
    # while warp 0 refills the 64-entry descriptor ring with later batches
    # (head_dim 64: a six-stage ring); every output is checked
    lens = np.random.default_rng(d + p).integers(1, 190, size=2000, endpoint=True)
    b = wl.custom_batch(lens, dtype="bf16", hq=32, hkv=8, d=d, p=p, seed=d + p, device="cuda")
    _run_batch(b, check_pool=False)


def test_eight_heads_cuda_cores_short_segments_past_the_descriptor_batches():
    # fp32 pools at eight heads per kv head (two CTAs per SM) with more than
    # 64 stages per CTA and a piece end at nearly every stage
    lens = np.random.default_rng(91).integers(1, 190, size=1200, endpoint=True)
    b = wl.custom_batch(lens, dtype="f32", hq=64, hkv=8, d=64, p=16, seed=91, device="cuda")
    _run_batch(b, check_pool=False)


def test_tensor_core_many_short_pieces():
    # eight heads per kv head over 2,000 short segments: about 150 one- or
    # two-stage pieces per CTA, so every Q buffer, descriptor slot and record
    # slot is reused many times; every output is checked
    lens = np.random.default_rng(77).integers(1, 190, size=2000, endpoint=True)
    b = wl.custom_batch(lens, dtype="bf16", hq=64, hkv=8, d=128, p=16, seed=77, device="cuda")
    _run_batch(b, check_pool=False)


def test_gqa8_tensor_core_decode_long():
    lens = np.array([40000, 3000, 65536, 1], np.int32)
    b = wl.custom_batch(lens, dtype="bf16", hq=32, hkv=4, d=128, p=16, seed=62, device="cuda")
    _run_batch(b)


def test_empty_batch_rows_and_all_empty():
    b = wl.custom_batch([0, 0, 5], dtype="bf16", hq=8, hkv=2, d=128, p=16, seed=5, device="cuda")
    _run_batch(b)
    b = wl.custom_batch([0, 0], dtype="bf16", hq=8, hkv=2, d=128, p=16, num_blocks=4, seed=6,
                        device="cuda")
    kc, vc = pu.device_pool(b)
    out, lse = pu.device_decode(b, kc, vc)
    assert not out.any() and np.isneginf(lse).all()


def test_llama_shaped_full_size():
    # the Llama-shaped decode layer at full size (64 sequences, 32/8 heads,
    # lengths 512..8192): whole pools bit for bit after the appends, every
    # row and head of the decode against the oracle
    b = wl.llama_batch(device="cuda")
    _run_batch(b)


@pytest.mark.parametrize("block_size", [16, 64])
def test_long_context_full_size(block_size):
    # the long-context decode at full size (8 sequences of 32k..64k rows):
    # whole pools, every row and head
    b = wl.long_batch(device="cuda", block_size=block_size)
    _run_batch(b)


def test_block_copy_bit_exact():
    b = wl.custom_batch([40, 70, 9], dtype="bf16", hq=8, hkv=2, d=128, p=16, seed=41,
                        device="cuda")
    kc, vc = pu.device_pool(b)
    pu.device_fill(b, kc, vc)
    hk, hv = pu.host_pool(b)
    pu.oracle_fill(b, hk, hv)
    used = set(b.block_tables[b.block_tables >= 0].tolist())
    free = [i for i in range(b.num_blocks) if i not in used]
    src = sorted(used)[:4]
    pairs = np.array(list(zip(src, free[:4])), np.int64)
    pkv.kv_block_copy(kc, vc, torch.from_numpy(pairs).cuda())
    assert oracle.kv_block_copy(hk, hv, pairs) == oracle.OK
    assert pkv.get_device_error() == 0
    assert pu.pools_equal_bytes(kc, hk) and pu.pools_equal_bytes(vc, hv)


def test_shared_prefix_cow_then_append_bit_exact():
    sp = wl.shared_prefix_batch(device="cuda", batch=16, prefix_len=256, shared_tail=8,
                                suffix_lo=16, suffix_hi=100, seed=51)
    shape = (sp.num_blocks, sp.block_size, sp.num_kv_heads, sp.head_dim)
    kc = torch.full(shape, float("nan"), dtype=torch.bfloat16, device="cuda")
    vc = torch.full_like(kc, float("nan"))
    pkv.kv_append(kc, vc, sp.parent_k, sp.parent_v, torch.from_numpy(sp.parent_slots).cuda())
    pkv.kv_block_copy(kc, vc, torch.from_numpy(sp.cow_pairs).cuda())
    pkv.kv_append(kc, vc, sp.child_k, sp.child_v, torch.from_numpy(sp.child_slots).cuda())
    hk = np.full(shape, 0x7FC0, np.uint16)
    hv = np.full(shape, 0x7FC0, np.uint16)
    n_par = sp.prefix_len + sp.shared_tail
    ps = np.array([oracle.slot_for_position(sp.parent_table, sp.block_size, t)
                   for t in range(n_par)], np.int64)
    oracle.kv_append(hk, hv, wl.to_numpy_storage(sp.parent_k), wl.to_numpy_storage(sp.parent_v), ps)
    oracle.kv_block_copy(hk, hv, sp.cow_pairs)
    ck, cv = wl.to_numpy_storage(sp.child_k), wl.to_numpy_storage(sp.child_v)
    for r in range(sp.num_seqs):
        table = np.concatenate([sp.prefix_block_ids, sp.suffix_tables[r]])
        lo, hi = sp.child_offsets[r], sp.child_offsets[r + 1]
        cs = np.array([oracle.slot_for_position(table, sp.block_size, n_par + i)
                       for i in range(hi - lo)], np.int64)
        oracle.kv_append(hk, hv, np.ascontiguousarray(ck[lo:hi]), np.ascontiguousarray(cv[lo:hi]), cs)
    torch.cuda.synchronize()
    assert pkv.get_device_error() == 0
    assert pu.pools_equal_bytes(kc, hk) and pu.pools_equal_bytes(vc, hv)


# ------------------------------------------------------------------ errors
def test_bad_slot_sets_error_and_writes_nothing():
    kc = torch.zeros(4, 16, 2, 64, dtype=torch.bfloat16, device="cuda")
    vc = torch.zeros_like(kc)
    k = torch.ones(3, 2, 64, dtype=torch.bfloat16, device="cuda")
    slots = torch.tensor([-1, 64, 5], dtype=torch.int64, device="cuda")
    pkv.kv_append(kc, vc, k, k, slots)
    assert pkv.get_device_error() == pkv.DEVERR_SLOT
    flat = kc.view(64, 2, 64)
    assert (flat[5] == 1).all() and (flat.sum() == 2 * 64)
    assert pkv.get_device_error() == 0  # read-and-clear


@pytest.mark.parametrize("hq", [8, 16])  # 16 / 2: eight heads per kv head, the tensor-core path
def test_bad_block_in_table_and_pair_set_error(hq):
    b = wl.custom_batch([40, 20], dtype="bf16", hq=hq, hkv=2, d=128, p=16, seed=61, device="cuda")
    kc, vc = pu.device_pool(b)
    pu.device_fill(b, kc, vc)
    bt = torch.from_numpy(b.block_tables).cuda()
    bt[0, 1] = b.num_blocks + 3
    sl = torch.from_numpy(b.seq_lens).cuda()
    pkv.paged_attention_decode(b.q, kc, vc, bt, sl, b.scale)
    assert pkv.get_device_error() & pkv.DEVERR_BLOCK
    pkv.kv_block_copy(kc, vc, torch.tensor([[0, -5]], dtype=torch.int64, device="cuda"))
    assert pkv.get_device_error() == pkv.DEVERR_BLOCK


@pytest.mark.parametrize("hq", [8, 16])
def test_length_beyond_table_sets_error(hq):
    b = wl.custom_batch([40, 20], dtype="bf16", hq=hq, hkv=2, d=128, p=16, seed=62, device="cuda")
    kc, vc = pu.device_pool(b)
    pu.device_fill(b, kc, vc)
    sl = torch.tensor([40, 10_000], dtype=torch.int32, device="cuda")
    pkv.paged_attention_decode(b.q, kc, vc, torch.from_numpy(b.block_tables).cuda(), sl, b.scale)
    assert pkv.get_device_error() & pkv.DEVERR_LENGTH


def test_host_validation_rejects_before_launch():
    kc = torch.zeros(4, 16, 2, 64, dtype=torch.bfloat16, device="cuda")
    q = torch.zeros(1, 6, 64, dtype=torch.bfloat16, device="cuda")  # 6 % 2 == 0 but G = 3
    bt = torch.zeros(1, 1, dtype=torch.int32, device="cuda")
    sl = torch.ones(1, dtype=torch.int32, device="cuda")
    with pytest.raises(pkv.PkvError) as ei:
        pkv.paged_attention_decode(q, kc, kc, bt, sl, 1.0)
    assert ei.value.status == pkv.PKV_ERR_UNSUPPORTED
    q = torch.zeros(1, 4, 64, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(pkv.PkvError) as ei:
        pkv.paged_attention_decode(q, kc, kc, bt, sl, 1.0, partition_size=24)
    assert ei.value.status == pkv.PKV_ERR_INVALID_ARG
    for p in (8, 24, 48, 80):  # block sizes the 32-row stages cannot tile
        kc3 = torch.zeros(4, p, 2, 64, dtype=torch.bfloat16, device="cuda")
        with pytest.raises(pkv.PkvError) as ei:
            pkv.paged_attention_decode(q, kc3, kc3, bt, sl, 1.0)
        assert ei.value.status == pkv.PKV_ERR_UNSUPPORTED
    assert pkv.get_device_error() == 0


# ------------------------------------------------------------------ allocator vs kernel blocks
@pytest.mark.parametrize("q", [1, 2, 4, 16])
def test_expand_block_tables_bit_exact(q):
    rng = np.random.default_rng(70 + q)
    t = rng.integers(0, 5000, size=(7, 33)).astype(np.int32)
    t[2, 10:] = -1
    t[5, :] = -1
    got = pkv.expand_block_tables(torch.from_numpy(t).cuda(), 16 * q, 16)
    torch.cuda.synchronize()
    assert pkv.get_device_error() == 0
    assert np.array_equal(got.cpu().numpy(), oracle.expand_table(t, q))


@pytest.mark.parametrize("pa,pk,hq", [(64, 16, 8), (256, 32, 16), (256, 16, 16)])
def test_decode_through_kernel_blocks(pa, pk, hq):
    """A pool of P_a-row allocator blocks decoded as P_k-row kernel blocks
    through the expanded tables (16 / 2 heads: the tensor-core path) equals
    the oracle's decode of the allocator-block view."""
    b = wl.custom_batch([700, 1, 129, 0, 2050, 64], dtype="bf16", hq=hq, hkv=2, d=128, p=pa,
                        seed=74, device="cuda")
    kc, vc = pu.device_pool(b)
    pu.device_fill(b, kc, vc)
    hk, hv = pu.host_pool(b)
    pu.oracle_fill(b, hk, hv)
    r = pa // pk
    view = (b.num_blocks * r, pk, b.num_kv_heads, b.head_dim)
    bt = pkv.expand_block_tables(torch.from_numpy(b.block_tables).cuda(), pa, pk)
    sl = torch.from_numpy(b.seq_lens).cuda()
    lse = torch.empty(b.num_seqs, b.num_q_heads, dtype=torch.float32, device="cuda")
    out = pkv.paged_attention_decode(b.q, kc.view(view), vc.view(view), bt, sl, b.scale, lse=lse)
    torch.cuda.synchronize()
    assert pkv.get_device_error() == 0
    ref, ref_lse = pu.oracle_decode(b, hk, hv)
    pu.assert_close(out.float().cpu().numpy(), ref, "kernel-block view out")
    pu.assert_close(lse.cpu().numpy(), ref_lse, "kernel-block view lse")


def test_expand_rejects_a_kernel_block_larger_than_the_allocator_block():
    t = torch.zeros(2, 3, dtype=torch.int32, device="cuda")
    for pa, pk in ((16, 32), (48, 32)):
        with pytest.raises(pkv.PkvError) as ei:
            pkv.expand_block_tables(t, pa, pk)
        assert ei.value.status == pkv.PKV_ERR_INVALID_ARG


# ------------------------------------------------------------------ churn trace
def test_churn_trace_small():
    """A short churn trace: requests finish and arrivals take blocks from the
    free FIFO, so stale rows of finished requests stay in the pool.  After
    every step (arrival prompts, then one row per request) the pools must
    equal the oracle's bit for bit, and every step's decode must match the
    oracle, which derives every slot itself from that step's block tables."""
    tr = wl.ChurnTrace(seed=44, concurrency=12, steps=10, median=60, sigma=1.0, cap=600,
                       mean_out=4)
    assert _churn(tr, hq=8, hkv=2, d=64, check_pools=True) >= 3  # the trace did churn


def test_churn_trace_config_shapes():
    """The churn trace at its configured width and heads (256 requests, 32/8
    heads, head_dim 128, lognormal prompts of median 1024), shorter outputs so
    that a dozen steps see arrivals: about 100 stages per CTA with piece ends
    among them.  Every step's output is checked against the oracle."""
    tr = wl.ChurnTrace(seed=45, concurrency=256, steps=12, median=1024, sigma=1.0, cap=4096,
                       mean_out=6)
    assert _churn(tr, hq=32, hkv=8, d=128, check_pools=False) >= 3


def test_churn_trace_as_configured():
    """The churn trace exactly as configured: 256 concurrent requests over 200
    decode steps, prompts lognormal (median 1024, sigma 1.0, capped at 16384),
    outputs geometric with mean 200, 32/8 heads, head_dim 128, block size 16,
    pool 1.25 x the dry run's peak.  Every step runs the arrivals' prompt
    appends, the step's append and the decode on the device, and the same
    appends in the oracle's own pool.  At ten evenly spaced steps the whole
    pools are compared bit for bit (every row appended since the last check,
    arrival prompts included, and every stale row of a freed block) and every
    row and head of that step's decode against the oracle."""
    tr = wl.ChurnTrace()  # the defaults are the configured trace
    assert (tr.concurrency, tr.steps, tr.block_size) == (256, 200, 16)
    checks = set(np.linspace(0, tr.steps - 1, 10).round().astype(int).tolist())
    assert len(checks) == 10
    assert _churn(tr, hq=32, hkv=8, d=128, check_pools=True, check_steps=checks,
                  fresh_q=True) >= 100


def _churn(tr, hq, hkv, d, check_pools, check_steps=None, fresh_q=False):
    """Run the trace on the device and in the oracle; returns the number of
    steps that saw arrivals.  check_steps: the steps whose pools and decode
    are compared (None: every step).  fresh_q: draw a new q every step."""
    p = tr.block_size
    B = tr.concurrency
    shape = (tr.num_blocks, p, hkv, d)
    kc = torch.full(shape, float("nan"), dtype=torch.bfloat16, device="cuda")
    vc = torch.full_like(kc, float("nan"))
    hk = np.full(shape, 0x7FC0, np.uint16)
    hv = np.full(shape, 0x7FC0, np.uint16)
    gen = wl.make_generator(44, "cuda")
    q = wl.randn((B, hq, d), "bf16", gen, "cuda")
    scale = 1.0 / np.sqrt(d)
    arrivals = 0
    for i_step, step in enumerate(tr.run()):
        if step.arrival_rows:
            arrivals += 1
            ak = wl.randn((step.arrival_rows, hkv, d), "bf16", gen, "cuda")
            av = wl.randn((step.arrival_rows, hkv, d), "bf16", gen, "cuda")
            pkv.kv_append(kc, vc, ak, av, torch.from_numpy(step.arrival_slots).cuda())
            slots = oracle.slots_for_positions(step.block_tables, p, step.arrival_seq_index,
                                               step.arrival_positions)
            assert oracle.kv_append(hk, hv, wl.to_numpy_storage(ak), wl.to_numpy_storage(av),
                                    slots) == oracle.OK
        nk = wl.randn((B, hkv, d), "bf16", gen, "cuda")
        nv = wl.randn((B, hkv, d), "bf16", gen, "cuda")
        pkv.kv_append(kc, vc, nk, nv, torch.from_numpy(step.step_slots).cuda())
        slots = oracle.slots_for_positions(step.block_tables, p, np.arange(B, dtype=np.int32),
                                           step.seq_lens.astype(np.int64) - 1)
        assert oracle.kv_append(hk, hv, wl.to_numpy_storage(nk), wl.to_numpy_storage(nv),
                                slots) == oracle.OK
        if fresh_q:
            q = wl.randn((B, hq, d), "bf16", gen, "cuda")
        bt = torch.from_numpy(step.block_tables).cuda()
        sl = torch.from_numpy(step.seq_lens).cuda()
        lse = torch.empty(B, hq, dtype=torch.float32, device="cuda")
        out = pkv.paged_attention_decode(q, kc, vc, bt, sl, scale, lse=lse)
        if check_steps is not None and i_step not in check_steps:
            continue
        torch.cuda.synchronize()
        assert pkv.get_device_error() == 0
        if check_pools:
            assert pu.pools_equal_bytes(kc, hk), f"K pool differs from the oracle's at step {i_step}"
            assert pu.pools_equal_bytes(vc, hv), f"V pool differs from the oracle's at step {i_step}"
        ref, ref_lse = oracle.paged_decode(wl.to_numpy_storage(q), hk, hv, step.block_tables,
                                           step.seq_lens, scale, nthreads=pu.NTHREADS)
        pu.assert_close(out.float().cpu().numpy(), ref, f"churn out, step {i_step}")
        pu.assert_close(lse.cpu().numpy(), ref_lse, f"churn lse, step {i_step}")
    torch.cuda.synchronize()
    assert pkv.get_device_error() == 0
    return arrivals


# ------------------------------------------------------------------ shared prefix
def _shared_prefix_run(sp, rows=None, suffix_lens=None, partition_size=0, block_offset=0):
    """Device: append parent rows, CoW copies, child rows, then the shared-prefix
    call.  Oracle: its own pool (own slots) and the concatenated-table decode.
    With block_offset, the device side alone relabels every block id i as
    i + block_offset in a pool that much larger (blocks below stay unused)."""
    shape = (sp.num_blocks, sp.block_size, sp.num_kv_heads, sp.head_dim)
    off, P = block_offset, sp.block_size

    def ids(x):
        return torch.from_numpy(np.where(x >= 0, x + off, x).astype(x.dtype)).cuda()

    def slots(x):
        return torch.from_numpy(np.where(x >= 0, x + off * P, x).astype(np.int64)).cuda()

    kc = torch.full((off + shape[0],) + shape[1:], float("nan"), dtype=torch.bfloat16, device="cuda")
    vc = torch.full_like(kc, float("nan"))
    pkv.kv_append(kc, vc, sp.parent_k, sp.parent_v, slots(sp.parent_slots))
    pkv.kv_block_copy(kc, vc, ids(sp.cow_pairs))
    pkv.kv_append(kc, vc, sp.child_k, sp.child_v, slots(sp.child_slots))
    lens = sp.suffix_lens if suffix_lens is None else np.asarray(suffix_lens, np.int32)
    lse = torch.empty(sp.num_seqs, sp.num_q_heads, dtype=torch.float32, device="cuda")
    out = pkv.shared_prefix_attention(
        sp.q, kc, vc, ids(sp.prefix_block_ids), sp.prefix_len,
        ids(sp.suffix_tables), torch.from_numpy(lens).cuda(), sp.scale,
        lse=lse, partition_size=partition_size)
    torch.cuda.synchronize()
    assert pkv.get_device_error() == 0
    hk = np.full(shape, 0x7FC0, np.uint16)
    hv = np.full(shape, 0x7FC0, np.uint16)
    n_par = sp.prefix_len + sp.shared_tail
    ps = np.array([oracle.slot_for_position(sp.parent_table, sp.block_size, t)
                   for t in range(n_par)], np.int64)
    oracle.kv_append(hk, hv, wl.to_numpy_storage(sp.parent_k), wl.to_numpy_storage(sp.parent_v), ps)
    oracle.kv_block_copy(hk, hv, sp.cow_pairs)
    ck, cv = wl.to_numpy_storage(sp.child_k), wl.to_numpy_storage(sp.child_v)
    for r in range(sp.num_seqs):
        table = np.concatenate([sp.prefix_block_ids, sp.suffix_tables[r]])
        lo, hi = sp.child_offsets[r], sp.child_offsets[r + 1]
        cs = np.array([oracle.slot_for_position(table, sp.block_size, n_par + i)
                       for i in range(hi - lo)], np.int64)
        oracle.kv_append(hk, hv, np.ascontiguousarray(ck[lo:hi]), np.ascontiguousarray(cv[lo:hi]), cs)
    q = wl.to_numpy_storage(sp.q)
    st, sl = sp.suffix_tables, lens
    if rows is not None:
        q, st, sl = q[rows], st[rows], sl[rows]
    ref, ref_lse = oracle.shared_prefix(np.ascontiguousarray(q), hk, hv, sp.prefix_block_ids,
                                        sp.prefix_len, np.ascontiguousarray(st),
                                        np.ascontiguousarray(sl), sp.scale, nthreads=pu.NTHREADS)
    got, got_lse = out.float().cpu().numpy(), lse.cpu().numpy()
    if rows is not None:
        got, got_lse = got[rows], got_lse[rows]
    pu.assert_close(got, ref, "shared prefix out")
    pu.assert_close(got_lse, ref_lse, "shared prefix lse")


@pytest.mark.parametrize("batch,prefix,hq,hkv,d", [
    (16, 256, 32, 8, 128), (5, 384, 8, 2, 128), (40, 128, 16, 16, 64), (3, 512, 16, 2, 128),
    (24, 256, 64, 8, 128),  # eight heads per kv head: the suffixes decode on the tensor cores
    # 2, 3 and 5 query tiles of 128 rows: odd tile counts leave a CTA's second
    # tile (B) partly or wholly past the last request
    (50, 256, 32, 8, 128), (80, 384, 32, 8, 128), (150, 256, 32, 8, 64),
])
def test_shared_prefix_small(batch, prefix, hq, hkv, d):
    sp = wl.shared_prefix_batch(device="cuda", batch=batch, prefix_len=prefix, shared_tail=8,
                                suffix_lo=8, suffix_hi=200, hq=hq, hkv=hkv, d=d, seed=81 + batch)
    _shared_prefix_run(sp)


@pytest.mark.parametrize("batch,prefix,hq,hkv,d,p", [
    (20, 256, 32, 8, 128, 32), (12, 512, 16, 4, 64, 64), (9, 512, 32, 8, 128, 128),
    (7, 512, 16, 2, 128, 256),
])
def test_shared_prefix_block_sizes(batch, prefix, hq, hkv, d, p):
    # the prefix kernel's 8-row-group boxes over blocks of 32 to 256 rows
    # (one box per block, or per 128-row slice of a larger one)
    sp = wl.shared_prefix_batch(device="cuda", batch=batch, prefix_len=prefix, shared_tail=8,
                                suffix_lo=8, suffix_hi=300, hq=hq, hkv=hkv, d=d, p=p,
                                seed=300 + batch + p)
    _shared_prefix_run(sp)


@pytest.mark.parametrize("hq", [32, 64])  # 64 / 8: the suffixes decode on the tensor cores
def test_shared_prefix_pool_past_2_31_elements(hq):
    """Every block the batch uses lies past element 2^31 of the pool: the
    prefix kernel's and the decode's block coordinates, and the CoW copy's
    and the appends' 64-bit offsets."""
    sp = wl.shared_prefix_batch(device="cuda", batch=24, prefix_len=512, shared_tail=8,
                                suffix_lo=8, suffix_hi=200, hq=hq, hkv=8, d=128, seed=211 + hq)
    off = 2**31 // (sp.block_size * sp.num_kv_heads * sp.head_dim) + 5
    _shared_prefix_run(sp, block_offset=off)


def test_shared_prefix_with_empty_suffixes():
    sp = wl.shared_prefix_batch(device="cuda", batch=9, prefix_len=256, shared_tail=0,
                                suffix_lo=0, suffix_hi=40, seed=91)
    lens = sp.suffix_lens.copy()
    lens[::3] = 0
    _shared_prefix_run(sp, suffix_lens=lens)


def test_shared_prefix_full_size():
    # 128 requests on one 2048-token prefix, every request and head
    sp = wl.shared_prefix_batch(device="cuda")
    _shared_prefix_run(sp)


@pytest.mark.parametrize("split_len", [0, 128, 384, 768, 896])
def test_prefix_states_per_split(split_len):
    """Each split's state equals the oracle's attention over that split's keys
    (splits of one to seven 128-key tiles; at 896 the one split is longer
    than the 768-key prefix)."""
    sp = wl.shared_prefix_batch(device="cuda", batch=20, prefix_len=768, shared_tail=0,
                                suffix_lo=1, suffix_hi=20, seed=95)
    shape = (sp.num_blocks, sp.block_size, sp.num_kv_heads, sp.head_dim)
    kc = torch.full(shape, float("nan"), dtype=torch.bfloat16, device="cuda")
    vc = torch.full_like(kc, float("nan"))
    pkv.kv_append(kc, vc, sp.parent_k, sp.parent_v, torch.from_numpy(sp.parent_slots).cuda())
    so, sl, split = pkv.prefix_attention_states(
        sp.q, kc, vc, torch.from_numpy(sp.prefix_block_ids).cuda(), sp.prefix_len, sp.scale,
        split_len=split_len)
    torch.cuda.synchronize()
    assert pkv.get_device_error() == 0 and split % 128 == 0
    hk = np.full(shape, 0x7FC0, np.uint16)
    hv = np.full(shape, 0x7FC0, np.uint16)
    ps = np.array([oracle.slot_for_position(sp.parent_table, sp.block_size, t)
                   for t in range(sp.prefix_len)], np.int64)
    oracle.kv_append(hk, hv, wl.to_numpy_storage(sp.parent_k)[:sp.prefix_len].copy(),
                     wl.to_numpy_storage(sp.parent_v)[:sp.prefix_len].copy(), ps)
    q = wl.to_numpy_storage(sp.q)
    n = -(-sp.prefix_len // split)
    for s in range(n):
        lo, hi = s * split, min((s + 1) * split, sp.prefix_len)
        ids = sp.prefix_block_ids[lo // sp.block_size: hi // sp.block_size]
        tables = np.tile(ids, (sp.num_seqs, 1)).astype(np.int32)
        lens = np.full(sp.num_seqs, hi - lo, np.int32)
        ref, ref_lse = oracle.paged_decode(q, hk, hv, tables, lens, sp.scale, nthreads=pu.NTHREADS)
        pu.assert_close(so[:, :, s].cpu().numpy(), ref, f"split {s} O")
        pu.assert_close(sl[:, :, s].cpu().numpy(), ref_lse, f"split {s} LSE")
