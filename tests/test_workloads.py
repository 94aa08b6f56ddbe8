"""The seeded input generators produce the structure each workload states
(CPU only; small shapes with the same recipes)."""
import torch

import workloads


def test_causal_mask_keeps_keys_up_to_the_query():
    M, N = 12, 5  # rows wrap around the square block: query = row mod N
    x = workloads.softmax_inputs(M, N, mask="causal", seed=3)["x"]
    for r in range(M):
        q = r % N
        assert torch.isfinite(x[r, :q + 1]).all()
        assert torch.isneginf(x[r, q + 1:]).all()


def test_keep_k_mask_keeps_k_distinct_columns_per_row():
    x = workloads.softmax_inputs(9, 300, dtype="bf16", mask="keep:7", seed=1)["x"]
    fin = torch.isfinite(x.float())
    assert (fin.sum(dim=1) == 7).all()
    assert (torch.isneginf(x.float()) | fin).all()
    # the mask is drawn after the samples: kept entries equal the unmasked draw
    ref = workloads.softmax_inputs(9, 300, dtype="bf16", seed=1)["x"]
    assert torch.equal(x[fin], ref[fin])


def test_shift_rows_and_spikes_counts():
    w = workloads.Workload("t", "softmax", 200, 64, "f32", "f32", sigma=1.0, shift_rows=2,
                           spikes_per_row=3)
    x = workloads.make(w)["x"]
    shifted = x.min(dim=1).values > 500
    assert int(shifted.sum()) == 2
    base = torch.where(shifted.unsqueeze(1), x - 1000.0, x)
    assert (base > 20).sum(dim=1).eq(3).all()  # N(0,1) samples never reach 20


def test_registered_workloads_are_consistent():
    for name, w in workloads.WORKLOADS.items():
        assert w.name == name
        assert w.M > 0 and w.N > 0
        assert w.min_bytes > 0
        if w.mask:
            assert w.op in ("softmax", "log_softmax", "logsumexp")
