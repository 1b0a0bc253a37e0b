"""Many verify steps back to back with programmatic dependent launch (the way the
bench runs them) against the same steps launched one kernel after another.

A race between overlapping kernels, or inside one, shows up only over many
consecutive launches: a wait that runs out sets the status word's timeout bit
and the decisions go wrong. 48 steps of an 8B-shape model (2 layers, the
attention in its 4 x 4-cluster layout at context 4096) must report a clean
status and give, step by step, the same accepted lengths, next tokens and
committed lengths as the serialized run.
"""
import numpy as np
import pytest

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
import synth  # noqa: E402
import synth.device as sd  # noqa: E402
import verify_step_02_b300 as vs  # noqa: E402

PAGE, GAMMA, C, STEPS = 16, 16, 4096, 48


def run(flags, wdev, shape, blocks):
    max_seq = C + STEPS * (GAMMA + 1) + 64
    table, n_pages = synth.contiguous_page_table([max_seq], PAGE, max_seq // PAGE + 1)
    ks, vs_ = sd.kv_pools(shape, n_pages, PAGE, torch.bfloat16, fill="normal")
    seq = torch.tensor([C], dtype=torch.int32, device="cuda")
    kv = vs.KVCache(ks, vs_, torch.from_numpy(table).cuda(), seq)
    model = vs.Model(vs.make_config(shape, vs.SV_BF16, 1, GAMMA, max_seq, PAGE, flags=flags), wdev)
    acc = torch.zeros(STEPS, dtype=torch.int32, device="cuda")
    nxt = torch.zeros(STEPS, dtype=torch.int32, device="cuda")
    committed = torch.zeros(STEPS, dtype=torch.int32, device="cuda")
    for i in range(STEPS):
        model.verify(blocks[i:i + 1], [GAMMA], kv, acc[i:i + 1], nxt[i:i + 1])
        committed[i:i + 1].copy_(seq)
    model.sync_status()   # raises on a timeout or a device check
    out = acc.cpu().numpy(), nxt.cpu().numpy(), committed.cpu().numpy()
    model.close()
    return out


def test_back_to_back_steps_match_serialized_launches():
    shape = dict(synth.SHAPES["8b"], n_layers=2)
    wdev = sd.random_bf16_model(shape)
    rng = np.random.default_rng(23)
    blocks = torch.from_numpy(rng.integers(0, shape["vocab"], size=(STEPS, GAMMA + 1)).astype(np.int32)).cuda()
    a = run(0, wdev, shape, blocks)
    b = run(vs.SV_FLAG_NO_PDL, wdev, shape, blocks)
    for x, y in zip(a, b):
        assert np.array_equal(x, y)
    assert (a[2] == C + np.cumsum(a[0] + 1)).all()
