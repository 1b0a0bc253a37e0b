"""The verify step captured once into a CUDA graph and replayed gives the same bits as direct calls.

The library's launches carry programmatic dependencies and take every per-call
choice on the host, so after one warm-up call a verify of a fixed batch shape
can be captured and replayed with new inputs copied into the captured buffers.
"""
import numpy as np
import pytest

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
import synth  # noqa: E402
import synth.device as sd  # noqa: E402
import verify_step_02_b300 as vs  # noqa: E402

PAGE = 16
GQA = dict(n_layers=2, d_model=512, n_heads=8, n_kv_heads=2, head_dim=128, ffn=1024, vocab=4096, rope_theta=1e6)


@pytest.mark.parametrize("kind", ["f32", "bf16"])
def test_graph_replay_equals_direct_calls(kind):
    shape = synth.SHAPES["tiny"] if kind == "f32" else GQA
    hw = synth.host_weights(shape, "f32" if kind == "f32" else "w12window")
    if kind == "bf16":  # moderate activations: the window weights scaled by 2^-4 (exact in bf16)
        for lay in hw["layers"]:
            for name in ("wqkv", "wo", "wgu", "wd"):
                lay[name] = (lay[name].astype(np.int64) - (4 << 7)).astype(np.uint16)
    wdev = sd.host_to_device_weights(hw, kind)
    dt = torch.float32 if kind == "f32" else torch.bfloat16
    B, gamma, C = 3, 6, 37
    cfg = vs.make_config(shape, vs.SV_F32 if kind == "f32" else vs.SV_BF16, B, gamma, 256, PAGE,
                         flags=vs.SV_FLAG_KEEP_LOGITS)
    lengths = [C + 4 * (gamma + 1) + 1] * B
    table, n_pages = synth.shuffled_page_table(lengths, PAGE, max(lengths) // PAGE + 2, 5, 5)
    rng = np.random.default_rng(17)
    blocks = [torch.from_numpy(rng.integers(0, shape["vocab"], size=(B, gamma + 1)).astype(np.int32)).cuda()
              for _ in range(4)]
    lens = [gamma, 2, 0]
    outs = []
    for mode in ("direct", "graph"):
        model = vs.Model(cfg, wdev)
        ks, vs_ = sd.kv_pools(shape, n_pages, PAGE, dt, fill="normal")
        seq = torch.full((B,), C, dtype=torch.int32, device="cuda")
        kv = vs.KVCache(ks, vs_, torch.from_numpy(table).cuda(), seq)
        tok = torch.zeros((B, gamma + 1), dtype=torch.int32, device="cuda")
        acc = torch.zeros(B, dtype=torch.int32, device="cuda")
        nxt = torch.zeros(B, dtype=torch.int32, device="cuda")
        res = []
        if mode == "direct":
            for blk in blocks:
                tok.copy_(blk)
                model.verify(tok, lens, kv, acc, nxt)
                res.append((model.logits(sum(l + 1 for l in lens)).clone(), acc.clone(), nxt.clone(), seq.clone()))
        else:
            tok.copy_(blocks[0])
            model.verify(tok, lens, kv, acc, nxt)       # warm-up call: first-use setup
            torch.cuda.synchronize()
            seq.fill_(C)
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g):
                model.verify(tok, lens, kv, acc, nxt)
            seq.fill_(C)
            for blk in blocks:
                tok.copy_(blk)
                g.replay()
                res.append((model.logits(sum(l + 1 for l in lens)).clone(), acc.clone(), nxt.clone(), seq.clone()))
        torch.cuda.synchronize()
        model.sync_status()
        outs.append(res)
        model.close()
    for (l1, a1, n1, s1), (l2, a2, n2, s2) in zip(*outs):
        assert torch.equal(l1, l2) and torch.equal(a1, a2) and torch.equal(n1, n2) and torch.equal(s1, s2)
