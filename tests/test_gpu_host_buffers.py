"""Host buffers: a call whose inputs (q, new K/V rows, positions, lengths,
block tables, expected tags) and outputs (out, flags) live in pinned host
memory, which the kernels read and write directly (no staging copy), gives
the same bytes as the call with device buffers: outputs, flags and the pool
after the append.  Covers pfkv_decode_step (separate and fused tag check),
the attention call on per-head tables, a BF16 pool, and a step graph whose
buffers are host memory; and pfkv_stage_copy, which stages a step's packed
host inputs into device memory with a kernel."""
import dataclasses

import pytest
import torch

from paged_fp8_kv_decode_gb300 import workloads as W
from test_gpu_parity import B  # noqa: F401  (fixture)

pytestmark = pytest.mark.gpu


def _db(spec):
    from paged_fp8_kv_decode_gb300.device_batch import DeviceBatch
    return DeviceBatch(W.make_batch(spec))


def _host(t):
    return None if t is None else t.detach().cpu().pin_memory()


def _host_pages(B, db):
    sb, sh = db.batch.len_strides
    tb, th = db.batch.bt_strides
    return B.Pages(db.spec.B, db.batch.max_pages, _host(db.block_tables), tb, th, _host(db.seq_lens),
                   sb, sh, _host(db.pages.expected_tags))


def _pool(db):
    c = db.cache
    return [t.clone() for t in (c.k_pages, c.v_pages, c.k_scale, c.v_scale) if t is not None]


def _restore(db, saved):
    c = db.cache
    for t, s in zip([t for t in (c.k_pages, c.v_pages, c.k_scale, c.v_scale) if t is not None], saved):
        t.copy_(s)


SPECS = {
    "llama8b": lambda: W.spec_llama8b("small"),
    "bf16": lambda: dataclasses.replace(W.spec_sweep(3, "bf16", scale="small"), append=True),
    "evict": lambda: W.spec_evict("small"),
}


@pytest.mark.parametrize("fused", [False, True])
@pytest.mark.parametrize("kind", sorted(SPECS))
def test_host_buffers_give_the_same_bytes(B, kind, fused):
    spec = SPECS[kind]()
    db = _db(spec)
    opt = B.PFKV_STAGE_FUSED_TAGS if fused else 0
    before = _pool(db)
    # device buffers
    if spec.append:
        B.pfkv_decode_step(db.cache, db.pages, db.positions, db.k_new, db.v_new, db.q, spec.sm_scale,
                           db.split_tokens, db.max_seq_len, db.workspace, db.out, db.flags,
                           append_flags=db.append_flags, options=opt)
    else:
        fn = B.pfkv_paged_decode_attn_fused_tags if fused else B.pfkv_paged_decode_attn
        fn(db.cache, db.pages, db.q, spec.sm_scale, db.split_tokens, db.max_seq_len, db.workspace,
           db.out, db.flags)
    torch.cuda.synchronize()
    want_out, want_flags, want_pool = db.out.clone(), db.flags.clone(), _pool(db)
    want_append = db.append_flags.clone() if spec.append else None
    # the same call with host buffers, from the same pool
    _restore(db, before)
    pages = _host_pages(B, db)
    q = _host(db.q)
    out = torch.full(db.out.shape, 7.0, dtype=db.out.dtype).pin_memory()
    flags = torch.full(db.flags.shape, 0xEE, dtype=db.flags.dtype).pin_memory()
    if spec.append:
        # append bits are OR-ed in (never cleared), so this buffer starts at zero
        append_flags = torch.zeros(db.append_flags.shape, dtype=db.append_flags.dtype).pin_memory()
        B.pfkv_decode_step(db.cache, pages, _host(db.positions), _host(db.k_new), _host(db.v_new), q,
                           spec.sm_scale, db.split_tokens, db.max_seq_len, db.workspace, out, flags,
                           append_flags=append_flags, options=opt)
    else:
        fn = B.pfkv_paged_decode_attn_fused_tags if fused else B.pfkv_paged_decode_attn
        fn(db.cache, pages, q, spec.sm_scale, db.split_tokens, db.max_seq_len, db.workspace, out, flags)
    torch.cuda.synchronize()
    assert torch.equal(out, want_out.cpu()), kind
    assert torch.equal(flags[:spec.B], want_flags.cpu()[:spec.B]), kind
    if spec.append:
        assert torch.equal(append_flags[:spec.B], want_append.cpu()[:spec.B]), kind
    for got, want in zip(_pool(db), want_pool):
        assert torch.equal(got, want), kind
    if kind == "evict":
        assert flags[:spec.B].any()  # stale tags flag requests through host-resident tags too


def test_step_graph_with_host_buffers(B):
    """A one-layer step graph captured with host pointers replays to the same
    bytes as direct calls with device buffers, twice (the second replay reads
    rewritten host inputs)."""
    spec = W.spec_llama8b("small")
    db = _db(spec)
    pages = _host_pages(B, db)
    q, kn, vn, pos = _host(db.q), _host(db.k_new), _host(db.v_new), _host(db.positions)
    out = torch.zeros(db.out.shape, dtype=db.out.dtype).pin_memory()
    flags = torch.zeros(db.flags.shape, dtype=db.flags.dtype).pin_memory()
    layer = B.Layer(db.cache, q, out, kn, vn, flags)
    g = B.pfkv_step_graph_create([layer], pages, pos, None, 1, db.append_flags, spec.Hq,
                                 spec.sm_scale, db.split_tokens, db.max_seq_len, db.workspace)
    for rnd in range(2):
        if rnd:
            q.mul_(-0.5)  # new host inputs for the second replay
            db.q.copy_(q)
        before = _pool(db)
        g.launch()
        torch.cuda.synchronize()
        got_out, got_flags, got_pool = out.clone(), flags.clone(), _pool(db)
        _restore(db, before)
        db.step()
        torch.cuda.synchronize()
        assert torch.equal(got_out, db.out.cpu()), rnd
        assert torch.equal(got_flags[:spec.B], db.flags.cpu()[:spec.B]), rnd
        for a, b in zip(got_pool, _pool(db)):
            assert torch.equal(a, b), rnd
    g.close()


def test_stage_copy_moves_bytes_between_host_and_device(B):
    g = torch.Generator().manual_seed(3)
    n = (1 << 20) + 48  # a multiple of 16, not of the kernel's grid
    host = torch.randint(0, 256, (n,), generator=g, dtype=torch.uint8).pin_memory()
    dev = torch.zeros(n, dtype=torch.uint8, device="cuda")
    B.pfkv_stage_copy(dev, host)
    back = torch.zeros(n, dtype=torch.uint8).pin_memory()
    dev2 = torch.zeros(n, dtype=torch.uint8, device="cuda")
    B.pfkv_stage_copy(dev2, dev)         # device to device
    B.pfkv_stage_copy(back, dev2)        # device to host
    B.pfkv_stage_copy(dev2, host, 0)     # nothing
    torch.cuda.synchronize()
    assert torch.equal(dev.cpu(), host) and torch.equal(back, host)


def test_staged_inputs_give_the_same_step(B):
    """A step whose packed inputs are staged from pinned host memory by
    pfkv_stage_copy, with out and flags in host memory, gives the bytes of the
    step on device inputs."""
    spec = W.spec_llama8b("small")
    db = _db(spec)
    db.pack_step_io()
    before = _pool(db)
    db.step()
    torch.cuda.synchronize()
    want_out, want_flags, want_pool = db.out.clone(), db.flags.clone(), _pool(db)
    _restore(db, before)
    h_in = db.io_in.detach().cpu().pin_memory()
    db.io_in.zero_()  # the staged copy must bring every input back
    out = torch.full(db.out.shape, 7.0, dtype=db.out.dtype).pin_memory()
    flags = torch.full(db.flags.shape, 0xEE, dtype=db.flags.dtype).pin_memory()
    B.pfkv_stage_copy(db.io_in, h_in)
    B.pfkv_decode_step(db.cache, db.pages, db.positions, db.k_new, db.v_new, db.q, spec.sm_scale,
                       db.split_tokens, db.max_seq_len, db.workspace, out, flags,
                       append_flags=db.append_flags)
    torch.cuda.synchronize()
    assert torch.equal(out, want_out.cpu())
    assert torch.equal(flags[:spec.B], want_flags.cpu()[:spec.B])
    for a, b in zip(_pool(db), want_pool):
        assert torch.equal(a, b)
