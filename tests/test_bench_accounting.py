"""The benchmark's work accounting (CPU only): algorithmic prefill FLOPs and
decode bytes against brute-force counts over positions, layers and windows."""
import bench
from synthetic import MODELS, WORKLOADS, Workload


def _pairs_brute(n, windows, L):
    tot = 0
    for l in range(L):
        w = windows[l] if windows is not None else 0
        for p in range(n):
            first = p + 1 - w if (w > 0 and p + 1 > w) else 0
            tot += p + 1 - first
    return tot


def test_prefill_flops_match_a_brute_force_count():
    m = MODELS["tiny"]
    proj_weights = sum(r * c for r, c in [(m.q_dim, m.d_model), (m.kv_dim, m.d_model), (m.kv_dim, m.d_model),
                                          (m.d_model, m.q_dim), (m.ffn_dim, m.d_model), (m.ffn_dim, m.d_model),
                                          (m.d_model, m.ffn_dim)])
    for windows in (None, (5, 0), (1, 40), (100, 100)):
        wl = Workload("t", m, 0, 0, 30, 1, layer_window=windows)
        for n in (0, 1, 7, 29):
            want = 2 * m.n_layers * proj_weights * n + 4 * m.n_heads * m.head_dim * _pairs_brute(n, windows, 2)
            assert bench.prefill_flops(wl, n) == want, (windows, n)


def test_decode_bytes_match_a_brute_force_count():
    wl = WORKLOADS["2.3b-32k-swa"]
    m = wl.model
    per_layer_pos = 2 * 2 * m.kv_dim
    for pos in (0, 4095, 4096, 20000):
        kv = 0
        for l in range(m.n_layers):
            w = wl.layer_window[l]
            kv += (min(pos + 1, w) if w > 0 else pos + 1) * per_layer_pos
        want = m.weight_bytes_per_token("fp16") + kv + m.n_layers * per_layer_pos
        assert wl.bytes_per_step(pos) == want


def test_prefill_flops_of_a_mixture_of_experts_count_the_router_and_the_active_experts():
    from synthetic import ModelConfig
    m = ModelConfig("m", 2, 64, 4, 2, 16, 96, 50, n_experts=6, top_k_experts=2)
    wl = Workload("m", m, 0, 0, 30, 1)
    attn = (64 * 64 + 2 * 32 * 64) + 64 * 64          # q, k, v and o projections
    ffn = 6 * 64 + 2 * (2 * 96 * 64 + 64 * 96)        # router rows + two experts' gate, up, down
    n = 11
    assert bench.prefill_flops(wl, n) == 2 * 2 * (attn + ffn) * n + 4 * 4 * 16 * _pairs_brute(n, None, 2)
