"""Whole-stack parity of the CUDA path against the CPU oracle, on the same
seeded inputs, plus invariants that hold on the GPU at any size."""

import numpy as np
import pytest

import synth
from parity import assert_parity, oracle_result, run_gpu, run_oracle, workload

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")

# Small stacks that still span several tiles, ragged row tails and GQA
# groups 3 and 4, for both head sizes.
RAGGED = {
    "ragged-hd64": synth.Dims(2, 512, 8, 2, 64, 1536, 130, 70, 1.0e4),
    "ragged-hd128": synth.Dims(3, 768, 6, 2, 128, 2048, 200, 37, 5.0e5),
    "single-row": synth.Dims(2, 256, 4, 2, 64, 768, 1, 5, 1.0e4),
    # q|k|v = 384+128+128 columns: the last 256-column QKV tile is half empty;
    # d = 384 takes the 128-column residual tiles
    "odd-heads": synth.Dims(2, 384, 3, 1, 128, 768, 77, 9, 1.0e4),
    # one row tile of 100 rows: every GEMM splits k over a cluster whose
    # CTAs finish row slices (four of 32 rows, the last ragged; down: eight
    # of 16 rows, the seventh ragged, the eighth empty)
    "row-split": synth.Dims(2, 512, 8, 2, 64, 1536, 100, 20, 1.0e4),
}


def _check(got, want, tag):
    assert_parity(got[0], want[0], f"{tag} hidden_out")
    for l in range(len(want[1])):
        assert_parity(got[1][l], want[1][l], f"{tag} k_rows[{l}]")
        assert_parity(got[2][l], want[2][l], f"{tag} v_rows[{l}]")


@pytest.mark.parametrize("name", ["tiny", "ragged-hd64", "ragged-hd128", "single-row", "odd-heads",
                                  "row-split"])
def test_small_stacks_match_oracle(name):
    dims = RAGGED.get(name) or synth.CONFIGS[name]
    dims, (layers, pk, pv, hidden) = workload(dims)
    want = oracle_result(dims)
    _check(run_gpu(dims, layers, pk, pv, hidden), want, name)


@pytest.mark.parametrize("name", ["llama3.2-1b", "llama3.2-3b-pp512",
                                  "llama3.2-3b-pp512-prefix1536"])
def test_full_size_stack_matches_oracle(name):
    dims, (layers, pk, pv, hidden) = workload(name)
    want = oracle_result(name)
    _check(run_gpu(dims, layers, pk, pv, hidden), want, name)


@pytest.mark.slow
def test_8b_stack_matches_oracle():
    """The 8B workload at its full batch (2048 rows over a 2048-row prefix),
    every row of the hidden output and of every layer's K/V rows against the
    oracle (a few minutes of float64 on the host)."""
    name = "llama3-8b-pp2048-prefix2048"
    dims, (layers, pk, pv, hidden) = workload(name)
    got = run_gpu(dims, layers, pk, pv, hidden)
    want = oracle_result(name)
    _check(got, want, name)


def test_causality_is_bitwise():
    dims, (layers, pk, pv, hidden) = workload(RAGGED["ragged-hd128"])
    j = 150
    h2 = hidden.copy()
    h2[j] += 1.0
    a = run_gpu(dims, layers, pk, pv, hidden)
    b = run_gpu(dims, layers, pk, pv, h2)
    assert np.array_equal(a[0][:j], b[0][:j])
    assert not np.array_equal(a[0][j:], b[0][j:])
    for l in range(dims.n_layers):
        assert np.array_equal(a[1][l][:j], b[1][l][:j])
        assert np.array_equal(a[2][l][:j], b[2][l][:j])


@pytest.mark.parametrize("name", ["ragged-hd64", "llama3.2-3b-pp512"])
def test_run_to_run_bitwise_determinism(name):
    """Split tiles are finished by whichever CTA arrives last; the sums, and
    so the results, must not depend on which one that is."""
    dims, (layers, pk, pv, hidden) = workload(RAGGED.get(name) or name)
    a = run_gpu(dims, layers, pk, pv, hidden)
    b = run_gpu(dims, layers, pk, pv, hidden)
    assert np.array_equal(a[0], b[0])
    for l in range(dims.n_layers):
        assert np.array_equal(a[1][l], b[1][l]) and np.array_equal(a[2][l], b[2][l])


def test_decode_equals_prefill_on_gpu():
    """B one-token calls at s, s+1, ... (each appending its K/V rows to the
    caches) give what one B-row call at s gives."""
    from dense_decoder_layer_gb300.stack import DenseStack
    dims = synth.CONFIGS["tiny"].replace(start_pos=3, batch=8)
    dims, (layers, pk, pv, hidden) = workload(dims)
    full = run_gpu(dims, layers, pk, pv, hidden)
    st = DenseStack(dims, dims.start_pos + dims.batch, 1)
    st.load_layers(layers)
    st.load_prefix(pk, pv)
    outs = []
    for b in range(dims.batch):
        outs.append(st.prefill(torch.from_numpy(hidden[b:b + 1].copy()), dims.start_pos + b).numpy())
    dec = np.concatenate(outs, 0).astype(np.float64)
    assert_parity(dec, full[0], "decode vs prefill hidden")
    from parity import bf16_to_f64
    for l in range(dims.n_layers):
        k, v = st.rows(l, dims.start_pos, dims.batch)
        assert_parity(bf16_to_f64(k), full[1][l], f"decode vs prefill k[{l}]")
        assert_parity(bf16_to_f64(v), full[2][l], f"decode vs prefill v[{l}]")
    want = run_oracle(dims, layers, pk, pv, hidden)
    assert_parity(dec, want[0], "decode vs oracle")
    st.close()


def test_device_io_call_matches_host_io_call():
    from dense_decoder_layer_gb300.stack import DenseStack
    dims, (layers, pk, pv, hidden) = workload(RAGGED["ragged-hd64"])
    host = run_gpu(dims, layers, pk, pv, hidden)
    st = DenseStack(dims, dims.start_pos + dims.batch, dims.batch)
    st.load_layers(layers)
    st.load_prefix(pk, pv)
    x = torch.from_numpy(hidden).cuda()
    out = torch.empty_like(x)
    st.prefill_device(x, dims.start_pos, out)
    st.sync()
    assert np.array_equal(out.cpu().numpy().astype(np.float64), host[0])
    st.prefill_device(x, dims.start_pos, x)  # in place
    st.sync()
    assert np.array_equal(x.cpu().numpy().astype(np.float64), host[0])
    st.close()
