"""Device-side input checks of the verify step, through the C ABI.

A bad token id, a page id outside the pool, or a block that runs past the
request's page table is recorded in the model's status word (read back by
sv_model_sync_status) instead of faulting: the offending rows are skipped
and every other request's results are exactly those of a clean run. The
failures are made on the host by passing such inputs; nothing here faults,
traps or hangs the GPU (every access the kernels make stays inside the
buffers: a flagged row writes no KV and reads no page).
"""
import numpy as np
import pytest

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
import synth  # noqa: E402
import synth.device as sd  # noqa: E402
import verify_step_02_b300 as vs  # noqa: E402

PAGE, GAMMA = 16, 4
SHAPES = {
    # float32 weights: the CUDA-core kernels
    "f32": synth.SHAPES["tiny"],
    # bf16 weights, GQA group 4: the tensor-core GEMM and attention
    "bf16": dict(n_layers=2, d_model=512, n_heads=8, n_kv_heads=2, head_dim=128, ffn=1024, vocab=4096,
                 rope_theta=1e6),
}


def setup(kind, ctx):
    shape = SHAPES[kind]
    hw = synth.host_weights(shape, "f32")
    wdev = sd.host_to_device_weights(hw, "f32")
    if kind == "bf16":
        wdev = {k: (v.to(torch.bfloat16) if torch.is_tensor(v) else [{n: t.to(torch.bfloat16) for n, t in lay.items()}
                                                                     for lay in v])
                for k, v in wdev.items()}
    dt = torch.float32 if kind == "f32" else torch.bfloat16
    cfg = vs.make_config(shape, vs.SV_F32 if kind == "f32" else vs.SV_BF16, len(ctx), GAMMA, 512, PAGE,
                         flags=vs.SV_FLAG_KEEP_LOGITS)
    model = vs.Model(cfg, wdev)
    lengths = [c + GAMMA + 1 for c in ctx]
    max_pages = max((n + PAGE - 1) // PAGE for n in lengths) + 1
    table, n_pages = synth.shuffled_page_table(lengths, PAGE, max_pages, 9, 1)
    return shape, model, table, n_pages, dt


def fresh_kv(shape, table, n_pages, dt, ctx):
    ks, vs_ = sd.kv_pools(shape, n_pages, PAGE, dt, fill="normal")
    # positions past each request's context start empty
    for r, c in enumerate(ctx):
        pos = np.arange(c, c + GAMMA + 1)
        for l in range(shape["n_layers"]):
            z = torch.zeros((len(pos), shape["n_kv_heads"], shape["head_dim"]))
            sd.write_positions(ks[l], table[r], pos, z, PAGE)
            sd.write_positions(vs_[l], table[r], pos, z, PAGE)
    seq = torch.tensor(ctx, dtype=torch.int32, device="cuda")
    return ks, vs_, seq


def step(model, shape, table, tok, kv_parts, lens):
    ks, vs_, seq = kv_parts
    kv = vs.KVCache(ks, vs_, torch.from_numpy(np.ascontiguousarray(table)).cuda(), seq)
    b = tok.shape[0]
    acc = torch.zeros(b, dtype=torch.int32, device="cuda")
    nxt = torch.zeros(b, dtype=torch.int32, device="cuda")
    model.verify(torch.from_numpy(tok).cuda(), lens, kv, acc, nxt)
    logits = model.logits(int(sum(lens) + b)).cpu().numpy()
    try:
        model.sync_status()
        status = vs.SV_OK, ""
    except vs.SvError as e:
        status = e.status, str(e)
    return acc.cpu().numpy(), nxt.cpu().numpy(), logits, seq.cpu().numpy(), status


@pytest.mark.parametrize("kind", ["f32", "bf16"])
def test_bad_token_and_bad_page_are_flagged_and_contained(kind):
    ctx = [40, 33, 70]
    shape, model, table, n_pages, dt = setup(kind, ctx)
    V = shape["vocab"]
    rng = np.random.default_rng(3)
    tok = rng.integers(0, V, size=(3, GAMMA + 1)).astype(np.int32)
    lens = [GAMMA] * 3
    clean_kv = fresh_kv(shape, table, n_pages, dt, ctx)
    acc0, nxt0, lg0, seq0, st0 = step(model, shape, table, tok, clean_kv, lens)
    assert st0[0] == vs.SV_OK, st0

    bad_tok = tok.copy()
    bad_tok[1, 2] = V + 7                          # request 1: a draft outside the vocabulary
    bad_table = table.copy()
    p2 = ctx[2] // PAGE                            # request 2: the page holding its block rows
    bad_table[2, p2] = n_pages + 3                 # ... now points past the pool
    kv = fresh_kv(shape, table, n_pages, dt, ctx)
    acc1, nxt1, lg1, seq1, st1 = step(model, shape, bad_table, bad_tok, kv, lens)
    assert st1[0] == vs.SV_ERR_DEVICE_CHECK, st1
    assert "token id out of range" in st1[1] and "page id out of range" in st1[1], st1[1]

    # request 0 is untouched: identical results and committed length
    rows = GAMMA + 1
    assert np.array_equal(lg1[:rows], lg0[:rows])
    assert (acc1[0], nxt1[0], seq1[0]) == (acc0[0], nxt0[0], seq0[0])
    # request 2's block rows wrote no KV anywhere: its original block slots are still empty,
    # and no page differs from the clean run except requests 1 and 2's block slots
    pos2 = np.arange(ctx[2], ctx[2] + rows)
    pos1 = np.arange(ctx[1], ctx[1] + rows)
    for l in range(shape["n_layers"]):
        got = sd.read_positions(kv[0][l], table[2], pos2, PAGE).float()
        assert not got[pos2 // PAGE == p2].any()
        a, b = kv[0][l].clone(), clean_kv[0][l].clone()
        for t, pos in ((table[1], pos1), (table[2], pos2)):
            sd.write_positions(a, t, pos, torch.zeros((rows, shape["n_kv_heads"], shape["head_dim"])), PAGE)
            sd.write_positions(b, t, pos, torch.zeros((rows, shape["n_kv_heads"], shape["head_dim"])), PAGE)
        assert torch.equal(a, b)
    model.close()


@pytest.mark.parametrize("kind", ["f32", "bf16"])
def test_block_past_the_page_table_is_a_capacity_error(kind):
    ctx = [40, 64]
    shape, model, table, n_pages, dt = setup(kind, ctx)
    rng = np.random.default_rng(4)
    tok = rng.integers(0, shape["vocab"], size=(2, GAMMA + 1)).astype(np.int32)
    lens = [GAMMA] * 2
    clean = step(model, shape, table, tok, fresh_kv(shape, table, n_pages, dt, ctx), lens)
    assert clean[4][0] == vs.SV_OK
    # request 1's context fills pages 0..3 exactly; a table of 4 columns has no page for its block
    short = np.ascontiguousarray(table[:, :4])
    assert (ctx[0] + GAMMA + 1 + PAGE - 1) // PAGE <= 4
    acc, nxt, lg, seq, st = step(model, shape, short, tok, fresh_kv(shape, table, n_pages, dt, ctx), lens)
    assert st[0] == vs.SV_ERR_KV_CAPACITY, st
    assert "past the request's page table" in st[1]
    rows = GAMMA + 1
    assert np.array_equal(lg[:rows], clean[2][:rows])
    assert (acc[0], nxt[0], seq[0]) == (clean[0][0], clean[1][0], clean[3][0])
    model.close()
