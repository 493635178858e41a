"""The five selective-scan workloads (shapes, dtypes, value ranges, seeds).

Distributions (all workloads): u, z, B, C, delta_raw ~ N(0, 1) iid;
D ~ N(0, 1); A[d, n] = -(n + 1); delta_bias = inverse softplus of dt,
dt log-uniform in ``dt_range``; dy ~ N(0, 1).  Seed = 1000 + index.
"""

TENSOR_IDS = {"u": 1, "delta": 2, "z": 3, "B": 4, "C": 5, "D": 6, "dt": 7, "dy": 8}

CONFIGS = [
    dict(index=0, name="tiny_f32", Bsz=2, Dch=16, L=64, N=16, dtype="f32",
         dt_range=(1e-3, 1e-1), mode="fwd", seed=1000),
    dict(index=1, name="mamba130m_layer_bf16", Bsz=8, Dch=1536, L=2048, N=16, dtype="bf16",
         dt_range=(1e-3, 1e-1), mode="fwd", seed=1001),
    dict(index=2, name="mamba370m_layer_f32_fwd_bwd", Bsz=8, Dch=2048, L=2048, N=16, dtype="f32",
         dt_range=(1e-3, 1e-1), mode="fwd_bwd", seed=1002),
    dict(index=3, name="long_seq_bf16", Bsz=1, Dch=5120, L=131072, N=16, dtype="bf16",
         dt_range=(1e-4, 1e-2), mode="fwd", seed=1003),
    dict(index=4, name="decode_step_bf16", Bsz=256, Dch=5120, L=1, N=16, dtype="bf16",
         dt_range=(1e-3, 1e-1), mode="step", steps=128, seed=1004),
]


def config(i: int) -> dict:
    return dict(CONFIGS[i])
