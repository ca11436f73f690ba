"""Step graphs: a decode step of several layers captured once and replayed
must give, layer by layer, exactly the bytes of the direct calls (same
kernels, same arguments), and must read the buffers' current contents on
every replay (new queries, new tokens, longer lengths).  Every replay is also
checked against the oracle stepping the same layers: pool bytes, scales and
flags bit for bit, outputs within the contract tolerance."""
import dataclasses

import numpy as np
import pytest
import torch

import oracle
from oracle_cases import assert_outputs_close, cache_dict, fill_pool, host_pool, pages_dict
from paged_fp8_kv_decode_gb300 import workloads as W
from test_gpu_parity import B  # noqa: F401  (fixture)

pytestmark = pytest.mark.gpu


def _layers(spec, batch, n, max_seq_len):
    from paged_fp8_kv_decode_gb300.device_batch import DeviceBatch
    T = int(batch.fill_lens.max())
    dbs = []
    for l in range(n):
        sl = dataclasses.replace(spec, seed=spec.seed + 100 * (l + 1))
        rows = (W.draw_kv_rows(sl, T, "k", device="cuda"), W.draw_kv_rows(sl, T, "v", device="cuda"))
        db = DeviceBatch(batch, rows=rows, q=W.draw_q(sl, device="cuda"), keep_rows=True)
        if spec.append:
            db.k_new.copy_(W.draw_new_token(sl, "k", device="cuda"))
            db.v_new.copy_(W.draw_new_token(sl, "v", device="cuda"))
        db.max_seq_len = max_seq_len  # room for the steps' growing lengths
        from paged_fp8_kv_decode_gb300 import binding as B
        need = B.pfkv_decode_workspace_size(db.cache, db.pages, spec.Hq, spec.split_tokens,
                                            max_seq_len)
        db.workspace = torch.empty(max(need, 256), dtype=torch.uint8, device="cuda")
        dbs.append(db)
    return dbs


def _same(a, b, label):
    for x, y in zip(a, b):
        assert torch.equal(x.out, y.out), label
        assert torch.equal(x.flags, y.flags), label
        assert np.array_equal(host_pool(x.cache.k_pages), host_pool(y.cache.k_pages)), label
        assert np.array_equal(host_pool(x.cache.v_pages), host_pool(y.cache.v_pages)), label
        if x.cache.k_scale is not None:
            assert torch.equal(x.cache.k_scale, y.cache.k_scale), label
            assert torch.equal(x.cache.v_scale, y.cache.v_scale), label
    # the graph's layers OR their append flags into layer 0's buffer; each
    # direct layer into its own
    want = a[0].append_flags.clone()
    for x in a[1:]:
        want |= x.append_flags
    assert torch.equal(want, b[0].append_flags), label


class OracleLayers:
    """The oracle's copy of every layer's pool, stepped like the GPU's: the
    fill from the layer's rows, then per step the append of that step's new
    token (kv_append with the tags checked) and the attention."""

    def __init__(self, spec, batch, dbs):
        self.spec, self.batch = spec, batch
        self.pools = []
        for d in dbs:
            k, v, ks, vs = fill_pool(spec, batch, W.bf16_bits(d.k_rows), W.bf16_bits(d.v_rows))
            self.pools.append((k, v, ks, vs))
        self.aflags = np.zeros(spec.B, np.uint8)  # OR over layers and steps

    def step(self, dbs, step, max_len):
        """Returns per layer (out, flags) of decode step `step` (positions and
        lengths grown by `step` tokens)."""
        spec, batch = self.spec, self.batch
        res = []
        for d, (k, v, ks, vs) in zip(dbs, self.pools):
            cache = cache_dict(spec, batch, k, v, ks, vs)
            pages = pages_dict(spec, batch, batch.seq_lens + step)
            if spec.append:
                fl = np.zeros(spec.B, np.uint8)
                oracle.kv_append(cache, pages, batch.positions + step, W.bf16_bits(d.k_new),
                                 W.bf16_bits(d.v_new), flags=fl)
                self.aflags |= fl
            res.append(oracle.paged_decode(cache, pages, W.bf16_bits(d.q), spec.Hq, spec.sm_scale,
                                           max_len))
        return res

    def compare(self, dbs, res, label):
        for l, (d, (k, v, ks, vs), (out, flags)) in enumerate(zip(dbs, self.pools, res)):
            lab = f"{label} layer {l}"
            assert np.array_equal(host_pool(d.cache.k_pages), k), lab
            assert np.array_equal(host_pool(d.cache.v_pages), v), lab
            if ks is not None:
                assert np.array_equal(d.cache.k_scale.cpu().numpy(), ks), lab
                assert np.array_equal(d.cache.v_scale.cpu().numpy(), vs), lab
            assert np.array_equal(d.flags.cpu().numpy()[:self.spec.B], flags), lab
            assert_outputs_close(d.out, out, lab)
        assert np.array_equal(dbs[0].append_flags.cpu().numpy()[:self.spec.B], self.aflags), label


@pytest.mark.parametrize("fused", [False, True])
@pytest.mark.parametrize("which", ["llama8b", "evict", "bf16"])
def test_graph_replays_equal_direct_calls(B, which, fused):
    if which == "llama8b":
        spec = W.spec_llama8b("small")
    elif which == "evict":
        spec = dataclasses.replace(W.spec_evict("small"), append=True)
    else:
        spec = dataclasses.replace(W.spec_sweep(3, "bf16", scale="small"), append=True,
                                   lens=np.array([300, 17, 999], np.int32))
    batch = W.make_batch(spec)
    n = 3
    max_len = int(batch.seq_lens.max()) + 40
    direct = _layers(spec, batch, n, max_len)
    graphed = _layers(spec, batch, n, max_len)
    ws = torch.empty(B.pfkv_decode_workspace_size(graphed[0].cache, graphed[0].pages, spec.Hq,
                                                  spec.split_tokens, max_len),
                     dtype=torch.uint8, device="cuda")
    g0 = graphed[0]
    layers = [B.Layer(cache=d.cache, q=d.q, out=d.out, k_new=d.k_new, v_new=d.v_new, flags=d.flags)
              for d in graphed]
    graph = B.pfkv_step_graph_create(layers, g0.pages, g0.positions, None, 1 if spec.append else 0,
                                     g0.append_flags, spec.Hq, spec.sm_scale, spec.split_tokens,
                                     max_len, ws, B.PFKV_STAGE_FUSED_TAGS if fused else 0)
    for d in direct:
        d.fused_tags = fused
    ref = OracleLayers(spec, batch, graphed)
    try:
        for step in range(3):
            if step:
                # next decode step: new queries and tokens, one more token per head
                for sets in (direct, graphed):
                    gen = torch.Generator(device="cuda").manual_seed(1000 + step)
                    for d in sets:
                        d.q.copy_(torch.randn(d.q.shape, generator=gen, device="cuda").to(torch.bfloat16))
                        if spec.append:
                            d.k_new.copy_(torch.randn(d.k_new.shape, generator=gen, device="cuda").to(torch.bfloat16))
                            d.v_new.copy_(torch.randn(d.v_new.shape, generator=gen, device="cuda").to(torch.bfloat16))
                        d.positions += 1
                        d.seq_lens += 1
            for d in direct:
                d.append_step()
                d.attend()
            graph.launch()
            torch.cuda.synchronize()
            _same(direct, graphed, f"{which} fused={fused} step {step}")
            ref.compare(graphed, ref.step(graphed, step, max_len), f"{which} fused={fused} step {step}")
            assert not graphed[0].flags[:spec.B].any() or spec.tags
    finally:
        graph.close()


def test_graph_reports_argument_errors_of_a_layer(B):
    spec = W.spec_llama8b("small")
    batch = W.make_batch(spec)
    d = _layers(spec, batch, 1, int(batch.seq_lens.max()))[0]
    bad = B.Layer(cache=d.cache, q=d.q, out=d.out, k_new=d.k_new, v_new=d.v_new, flags=d.flags)
    with pytest.raises(B.PfkvError) as e:  # group size 3 is unsupported
        B.pfkv_step_graph_create([bad], d.pages, d.positions, None, 1, d.append_flags, 24,
                                 spec.sm_scale, 0, d.max_seq_len, d.workspace)
    assert e.value.status == 2
