"""Prefill and autoregressive decoding through the verify step's kernels (sv_prefill), against the oracle.

- tiny fp32 (CUDA-core kernels): a 64-token prompt fed as four 16-row blocks;
  the cached K/V of every position, the last block's logits and the greedy
  token after the prompt match the oracle's prefill; then 8 one-row steps
  reproduce the oracle's autoregressive greedy continuation.
- bf16 GQA (tensor-core kernels): one long block of 100 rows (400 attention
  rows per kv head, four 128-row tiles) after a 40-position context, batched
  with a 37-row block; every logit and the written K/V match the oracle.
"""
import numpy as np
import pytest

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
import synth  # noqa: E402
import synth.device as sd  # noqa: E402
import verify_step_02_b300 as vs  # noqa: E402
from oracle import decoder, spec  # noqa: E402

from helpers import LOGIT_TOL, classify_greedy, oracle_weights, report_decisions  # noqa: E402

PAGE = 16


def _kv(shape, lengths, kind, max_pages):
    table, n_pages = synth.contiguous_page_table(lengths, PAGE, max_pages)
    dt = torch.float32 if kind == "f32" else torch.bfloat16
    ks, vs_ = sd.kv_pools(shape, n_pages, PAGE, dt, fill="zeros")
    return ks, vs_, table


def test_tiny_prefill_in_blocks_then_ar_decode():
    shape = synth.SHAPES["tiny"]
    hw = synth.host_weights(shape, "f32")
    cfg, W = oracle_weights(shape, hw, "f32")
    prompt = [int(x) for x in synth.uniform_tokens(64, cfg.vocab, 1, 0)]
    st, lo, nk, nv = spec.prefill(cfg, W, prompt)
    n_o = int(np.argmax(lo[-1]))
    gamma = 15
    model = vs.Model(vs.make_config(shape, vs.SV_F32, 1, gamma, 128, PAGE, flags=vs.SV_FLAG_KEEP_LOGITS),
                     sd.host_to_device_weights(hw, "f32"))
    ks, vs_, table = _kv(shape, [96], "f32", 8)
    seq = torch.zeros(1, dtype=torch.int32, device="cuda")
    kv = vs.KVCache(ks, vs_, torch.from_numpy(table).cuda(), seq)
    nxt = torch.zeros(1, dtype=torch.int32, device="cuda")
    tok = torch.zeros((1, gamma + 1), dtype=torch.int32, device="cuda")
    for b0 in range(0, 64, gamma + 1):
        tok.copy_(torch.tensor([prompt[b0:b0 + gamma + 1]], dtype=torch.int32))
        model.prefill(tok, [gamma], kv, nxt)
    lg = model.logits(gamma + 1).cpu().numpy().astype(np.float64)
    model.sync_status()
    assert int(seq.item()) == 64
    assert np.abs(lg - lo[48:64]).max() <= LOGIT_TOL["f32"]
    pos = np.arange(64)
    for l in range(shape["n_layers"]):
        assert np.allclose(sd.read_positions(ks[l], table[0], pos, PAGE).cpu().numpy(), nk[l], rtol=1e-5, atol=1e-5)
        assert np.allclose(sd.read_positions(vs_[l], table[0], pos, PAGE).cpu().numpy(), nv[l], rtol=1e-5, atol=1e-5)
    report_decisions("tiny prefill next token", [classify_greedy(lo[-1:], [], 0, int(nxt.item()))], 0)
    # autoregressive greedy, one row per step, from the oracle's committed state
    spec.commit(st, [], [a[-1:] for a in nk], [a[-1:] for a in nv], 0, n_o)
    ar = spec.ar_greedy(cfg, W, st, 8)
    got = [int(nxt.item())]
    for _ in range(8):
        tok[0, 0] = got[-1]
        model.prefill(tok, [0], kv, nxt)
        got.append(int(nxt.item()))
    model.sync_status()
    assert got == ar.emitted[:9], (got, ar.emitted)
    assert int(seq.item()) == 72
    model.close()


def test_bf16_long_blocks_over_several_row_tiles():
    shape = dict(n_layers=2, d_model=512, n_heads=8, n_kv_heads=2, head_dim=128, ffn=1024, vocab=4096,
                 rope_theta=1e6)
    hw = synth.host_weights(shape, "w12window")
    for lay in hw["layers"]:  # moderate activations: the window weights scaled by 2^-4 (exact in bf16)
        for name in ("wqkv", "wo", "wgu", "wd"):
            lay[name] = (lay[name].astype(np.int64) - (4 << 7)).astype(np.uint16)
    cfg, W = oracle_weights(shape, hw, "bf16")
    rng = np.random.default_rng(21)
    ctx, lens = [40, 7], [99, 36]
    states = []
    for r, c in enumerate(ctx):
        stt = spec.empty_state(cfg, int(rng.integers(0, cfg.vocab)), request_id=r)
        stt.k = [decoder.round_to_bf16(rng.standard_normal((c, 2, 128))) for _ in range(2)]
        stt.v = [decoder.round_to_bf16(rng.standard_normal((c, 2, 128))) for _ in range(2)]
        states.append(stt)
    blocks = [[int(x) for x in rng.integers(0, cfg.vocab, size=n + 1)] for n in lens]
    gamma = 127
    wdev = sd.host_to_device_weights(hw, "bf16")
    model = vs.Model(vs.make_config(shape, vs.SV_BF16, 2, gamma, 256, PAGE, flags=vs.SV_FLAG_KEEP_LOGITS), wdev)
    lengths = [c + n + 1 for c, n in zip(ctx, lens)]
    max_pages = max((n + PAGE - 1) // PAGE for n in lengths) + 1
    table, n_pages = synth.shuffled_page_table(lengths, PAGE, max_pages, 5, 5)
    ks, vs_ = sd.kv_pools(shape, n_pages, PAGE, torch.bfloat16, fill="zeros")
    for r, stt in enumerate(states):
        for l in range(shape["n_layers"]):
            sd.write_positions(ks[l], table[r], np.arange(ctx[r]), torch.from_numpy(stt.k[l]), PAGE)
            sd.write_positions(vs_[l], table[r], np.arange(ctx[r]), torch.from_numpy(stt.v[l]), PAGE)
    seq = torch.tensor(ctx, dtype=torch.int32, device="cuda")
    kv = vs.KVCache(ks, vs_, torch.from_numpy(table).cuda(), seq)
    tok = np.zeros((2, gamma + 1), np.int32)
    for r, blk in enumerate(blocks):
        tok[r, :len(blk)] = blk
    nxt = torch.zeros(2, dtype=torch.int32, device="cuda")
    model.prefill(torch.from_numpy(tok).cuda(), lens, kv, nxt)
    lg = model.logits(sum(lens) + 2).cpu().numpy().astype(np.float64)
    model.sync_status()
    assert np.array_equal(seq.cpu().numpy(), np.array(ctx) + np.array(lens) + 1)
    row = 0
    verdicts = []
    for r, stt in enumerate(states):
        lo, nk, nv = decoder.forward_block(cfg, W, stt.k, stt.v, blocks[r], ctx[r])
        rows = lens[r] + 1
        err = np.abs(lg[row:row + rows] - lo).max()
        print(f"[prefill bf16] request {r}: {rows} rows, max |dlogit| {err:.4f}")
        assert err <= LOGIT_TOL["bf16"], (r, err)
        verdicts.append(classify_greedy(lo[-1:], [], 0, int(nxt[r].item())))
        pos = ctx[r] + np.arange(rows)
        for l in range(shape["n_layers"]):
            gk = sd.read_positions(ks[l], table[r], pos, PAGE).float().cpu().numpy()
            gv = sd.read_positions(vs_[l], table[r], pos, PAGE).float().cpu().numpy()
            assert np.allclose(gk, nk[l], rtol=2 ** -7, atol=1e-2)
            assert np.allclose(gv, nv[l], rtol=2 ** -7, atol=1e-2)
        row += rows
    report_decisions("bf16 long-block prefill next tokens", verdicts, 1)
    model.close()
