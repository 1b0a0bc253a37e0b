"""GPU verify step against the oracle at the full 8B-class and 27B-class sizes.

8B-class: 36 layers, d 4096, 32 q / 8 kv heads x 128, ffn 12288, vocab 151936,
bf16 N(0, 0.02); random bf16 N(0, 1) context of 4096; one request with 16
drafts (M = 17), temperature 0. Every logit of the block is compared.

27B-class: 64 layers, d 5120, 40 q / 8 kv heads x 128, ffn 17408, vocab
151936; 32 requests with contexts uniform in 512..8192 on a shuffled pool of
16-token pages; verify lengths from the cumulative-confidence rule
(c_i ~ Beta(8, 2), keep while prod c >= 0.3). The oracle recomputes requests
0, 7 and 31 through all layers (the others are checked through the commit).
"""
import numpy as np
import pytest

pytestmark = [pytest.mark.gpu, pytest.mark.slow]

torch = pytest.importorskip("torch")
import synth  # noqa: E402
import synth.device as sd  # noqa: E402
import verify_step_02_b300 as vs  # noqa: E402
from oracle import decoder  # noqa: E402

from helpers import LOGIT_TOL, DeviceContext, device_oracle_weights, classify_greedy  # noqa: E402

PAGE = 16


def _verify(model, tokens, lens, kv, gamma):
    b = len(lens)
    tok = np.zeros((b, gamma + 1), np.int32)
    for r, t in enumerate(tokens):
        tok[r, :len(t)] = t
    acc = torch.zeros(b, dtype=torch.int32, device="cuda")
    nxt = torch.zeros(b, dtype=torch.int32, device="cuda")
    model.verify(torch.from_numpy(tok).cuda(), lens, kv, acc, nxt)
    m = int(sum(l + 1 for l in lens))
    logits = model.logits(m)
    model.sync_status()
    return acc.cpu().numpy(), nxt.cpu().numpy(), logits


def test_8b_gamma16_block_matches_oracle():
    shape = synth.SHAPES["8b"]
    C, gamma = 4096, 16
    wdev = sd.random_bf16_model(shape)
    table, n_pages = synth.contiguous_page_table([C + gamma + 1], PAGE, (C + gamma + 1) // PAGE + 2)
    ks, vs_ = sd.kv_pools(shape, n_pages, PAGE, torch.bfloat16, fill="normal")
    seq = torch.tensor([C], dtype=torch.int32, device="cuda")
    kv = vs.KVCache(ks, vs_, torch.from_numpy(table).cuda(), seq)
    rng = np.random.default_rng(2)
    block = [int(x) for x in rng.integers(0, shape["vocab"], size=gamma + 1)]
    ctx = DeviceContext(ks, table[0], C, PAGE), DeviceContext(vs_, table[0], C, PAGE)
    cfg, W = device_oracle_weights(shape, wdev)
    lo, nk, nv = decoder.forward_block(cfg, W, ctx[0], ctx[1], block, C, rowwise=False)
    model = vs.Model(vs.make_config(shape, vs.SV_BF16, 1, gamma, C + 64, PAGE, flags=vs.SV_FLAG_KEEP_LOGITS), wdev)
    acc, nxt, lg = _verify(model, [block], [gamma], kv, gamma)
    lg = lg.cpu().numpy().astype(np.float64)
    err = np.abs(lg - lo).max()
    assert err <= LOGIT_TOL["bf16"], err
    assert classify_greedy(lo, block[1:], acc[0], nxt[0]) in ("match", "near_tie")
    assert int(seq.item()) == C + int(acc[0]) + 1
    pos = C + np.arange(gamma + 1)
    for l in (0, shape["n_layers"] - 1):
        gk = sd.read_positions(ks[l], table[0], pos, PAGE).float().cpu().numpy()
        gv = sd.read_positions(vs_[l], table[0], pos, PAGE).float().cpu().numpy()
        assert np.allclose(gk, nk[l], rtol=2 ** -7, atol=1e-2)
        assert np.allclose(gv, nv[l], rtol=2 ** -7, atol=1e-2)
    model.close()


def test_27b_ragged_batch32_shuffled_pages():
    shape = synth.SHAPES["27b"]
    B, gamma = 32, 16
    rng = np.random.default_rng(3)
    ctx_len = rng.integers(512, 8193, size=B)
    lens = synth.truncated_verify_lens(B, gamma, 0.3, 3, 1)
    wdev = sd.random_bf16_model(shape)
    need = [int(c) + gamma + 1 for c in ctx_len]
    max_pages = max((n + PAGE - 1) // PAGE for n in need) + 1
    table, n_pages = synth.shuffled_page_table(need, PAGE, max_pages, 3, 2)
    ks, vs_ = sd.kv_pools(shape, n_pages, PAGE, torch.bfloat16, fill="normal")
    seq = torch.tensor(ctx_len, dtype=torch.int32, device="cuda")
    kv = vs.KVCache(ks, vs_, torch.from_numpy(table).cuda(), seq)
    blocks = [[int(x) for x in rng.integers(0, shape["vocab"], size=int(l) + 1)] for l in lens]
    model = vs.Model(vs.make_config(shape, vs.SV_BF16, B, gamma, 8192 + gamma + 16, PAGE,
                                    flags=vs.SV_FLAG_KEEP_LOGITS), wdev)
    acc, nxt, lg = _verify(model, blocks, [int(l) for l in lens], kv, gamma)
    assert np.array_equal(seq.cpu().numpy(), ctx_len + acc + 1)
    row0 = np.r_[0, np.cumsum(np.asarray(lens) + 1)]
    picks = [0, 7, 31]
    cfg, W = device_oracle_weights(shape, wdev)
    reqs = [(DeviceContext(ks, table[r], int(ctx_len[r]), PAGE), DeviceContext(vs_, table[r], int(ctx_len[r]), PAGE),
             blocks[r], int(ctx_len[r])) for r in picks]
    outs = decoder.forward_blocks(cfg, W, reqs, rowwise=False)
    for r, (lo, _, _) in zip(picks, outs):
        g = lg[row0[r]:row0[r + 1]].cpu().numpy().astype(np.float64)
        err = np.abs(g - lo).max()
        assert err <= LOGIT_TOL["bf16"], (r, err)
        assert classify_greedy(lo, blocks[r][1:], acc[r], nxt[r]) in ("match", "near_tie")
    model.close()
