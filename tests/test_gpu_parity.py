"""GPU parity: liblowbit's CUDA kernels against the fp64 CPU oracle.

Packing and unpacking must be bit-exact.  The layer output must meet the
tolerance in tests/parity.py.  Small cases run the oracle on every output;
the full Llama-shaped layers run it on sampled output rows.
"""
import numpy as np
import pytest
import torch

import oracle
import synth
from parity import DeviceLayer, check_close, y_to_f64

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():  # collected on CPU machines too; every test here is gpu-marked
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

import bit_groupwise_weight_gb300 as lb  # noqa: E402
from bit_groupwise_weight_gb300 import build as lbuild  # noqa: E402

lbuild.build()
ORACLE = oracle.Oracle()
PATHS = [lb.PATH_QMV, lb.PATH_QMM]
PATH_IDS = {lb.PATH_QMV: "qmv", lb.PATH_QMM: "qmm"}


# ---------------------------------------------------------------------------
# Packing (bit-exact).
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("bits", range(1, 8))
@pytest.mark.parametrize("N,K", [(1, 8), (3, 32), (17, 96), (5, 256), (64, 4096), (7, 14336)])
def test_pack_bit_exact(bits, N, K):
    r = np.random.default_rng(bits * 1000 + N + K)
    codes = r.integers(0, 256, size=(N, K), dtype=np.uint8)   # high bits must be ignored
    got = lb.pack_weights(torch.from_numpy(codes).cuda(), bits).cpu().numpy()
    assert np.array_equal(got, ORACLE.pack(codes, bits))


@pytest.mark.parametrize("bits", range(1, 8))
@pytest.mark.parametrize("N,K", [(1, 8), (17, 96), (64, 4096)])
def test_unpack_bit_exact(bits, N, K):
    r = np.random.default_rng(bits * 7 + N)
    packed = r.integers(0, 256, size=(N, K * bits // 8), dtype=np.uint8)
    got = lb.unpack_weights(torch.from_numpy(packed).cuda(), K, bits).cpu().numpy()
    assert np.array_equal(got, ORACLE.unpack(packed, K, bits))


def test_pack_full_size_gate_up_7bit():
    # 8B gate+up at b = 7: 117 M codes -> 103 MB.  Sampled rows against the oracle,
    # the whole matrix against the kernel's own unpack.
    N, K, bits = 28672, 4096, 7
    codes = synth.make_codes(0, N, K, bits)
    dc = torch.from_numpy(codes).cuda()
    packed = lb.pack_weights(dc, bits)
    assert torch.equal(lb.unpack_weights(packed, K, bits), dc)
    rows = np.random.default_rng(1).choice(N, 64, replace=False)
    assert np.array_equal(packed[torch.from_numpy(rows).cuda()].cpu().numpy(),
                          ORACLE.pack(codes[rows], bits))


# ---------------------------------------------------------------------------
# The layer, small shapes: every output against the oracle.
# ---------------------------------------------------------------------------

def _oracle_y(L):
    return ORACLE.linear(L.x, ORACLE.pack(L.codes, L.bits), L.scales, L.zeros, L.bias,
                         L.K, L.bits, L.group)


@pytest.mark.parametrize("path", PATHS, ids=lambda p: PATH_IDS[p])
@pytest.mark.parametrize("bits", range(1, 8))
@pytest.mark.parametrize("group", [32, 64, 128, 256])
def test_linear_small_every_bits_group(path, bits, group):
    L = synth.make_layer(10 + bits, 1, 4 * 256, 131, bits, group, bias=(bits % 2 == 1))
    d = DeviceLayer(L)
    check_close(y_to_f64(d.run(path)), _oracle_y(L), f"b={bits} g={group}")


@pytest.mark.parametrize("path", PATHS, ids=lambda p: PATH_IDS[p])
@pytest.mark.parametrize("M", [1, 2, 3, 4, 5, 8, 16, 17, 32, 33, 64, 130])
def test_linear_small_every_m(path, M):
    L = synth.make_layer(20 + M, M, 640, 257, 5, 64, bias=True, outliers=True)
    d = DeviceLayer(L)
    check_close(y_to_f64(d.run(path)), _oracle_y(L), f"M={M}")


@pytest.mark.parametrize("path", PATHS, ids=lambda p: PATH_IDS[p])
@pytest.mark.parametrize("M,K,N,bits,group", [
    (1, 32, 1, 3, 32),          # smallest K = g = 32, one output
    (1, 32, 7, 7, 32),
    (2, 64, 3, 1, 64),
    (3, 96, 5, 6, 32),          # K not a multiple of 128
    (1, 4096 + 32, 33, 4, 32),  # ragged K tail over the CTA's stride
    (4, 14336, 40, 2, 128),     # long K
    (1, 256, 1000, 3, 256),     # ragged N
])
def test_linear_edge_shapes(path, M, K, N, bits, group):
    L = synth.make_layer(30 + K + N, M, K, N, bits, group, bias=True)
    d = DeviceLayer(L)
    if path == lb.PATH_QMM and K % 128 != 0:
        # The tensor-core kernel takes K in steps of 128 codes; it refuses other shapes.
        with pytest.raises(lb.LowbitError) as e:
            d.run(path)
        assert e.value.status == 2
        return
    check_close(y_to_f64(d.run(path)), _oracle_y(L), f"{(M, K, N, bits, group)}")


@pytest.mark.parametrize("bits", range(1, 8))
@pytest.mark.parametrize("M,K,N,group", [
    (1, 2048, 10007, 64),       # three 16-row tiles per CTA, the last one ragged
    (2, 3072, 5003, 128),       # two rows of x, K not a power of two
    (1, 8192, 4999, 256),       # K split into chunks per stage
    (2, 1024, 9001, 32),        # smallest K the decode kernel takes, g = 32
])
def test_linear_decode_tiles_and_chunks(bits, M, K, N, group):
    L = synth.make_layer(60 + bits + K, M, K, N, bits, group, bias=(M == 2), outliers=(M == 2))
    d = DeviceLayer(L)
    check_close(y_to_f64(d.run(lb.PATH_QMV)), _oracle_y(L), f"{(M, K, N, bits, group)}")


# Rows of x per launch of the tensor-core decode kernel: 2 (g = 32), 4 (g = 64),
# 8 (g >= 128).  K = 1280 (five 256-code slices, one CTA) and ragged N = 203 take
# that kernel; M runs through every column-set variant and one launch past the
# limit (two launches).
_ROWS = {32: 2, 64: 4, 128: 8, 256: 8}


@pytest.mark.parametrize("bits", [1, 3, 4, 7])
@pytest.mark.parametrize("group", [32, 64, 128, 256])
def test_decode_kernel_rows_per_launch(bits, group):
    for M in sorted({1, 2, _ROWS[group] // 2 + 1, _ROWS[group], _ROWS[group] + 1}):
        L = synth.make_layer(70 + bits + M, M, 1280, 203, bits, group, bias=True, outliers=True)
        d = DeviceLayer(L)
        check_close(y_to_f64(d.run(lb.PATH_QMV)), _oracle_y(L), f"M={M} b={bits} g={group}")


@pytest.mark.parametrize("M,K,N,bits,group", [
    (8, 12288, 77, 5, 128),     # K over a cluster of 3 CTAs, eight rows of x
    (4, 8192, 45, 2, 64),       # cluster of 2, four rows, two column sets
    (1, 32768, 40, 7, 256),     # the longest K: a cluster of 8
    (3, 14336, 33, 6, 32),      # g = 32: two launches of the cluster kernel
])
def test_decode_kernel_cluster_rows(M, K, N, bits, group):
    L = synth.make_layer(90 + M + bits, M, K, N, bits, group, bias=True, outliers=True)
    d = DeviceLayer(L)
    check_close(y_to_f64(d.run(lb.PATH_QMV)), _oracle_y(L), f"{(M, K, N, bits, group)}")


def test_linear_single_qmv_full():
    # K = N = 4096, M = 1, b = 4, g = 64, seed 0: every output.
    L = synth.make_layer(0, **synth.SINGLE_QMV)
    d = DeviceLayer(L)
    check_close(y_to_f64(lb.linear(d.x, d.packed, d.scales, d.zeros, None, 4, 64)), _oracle_y(L))


def test_empty_calls_write_nothing():
    x = torch.zeros((0, 64), dtype=torch.bfloat16, device="cuda")
    w = torch.zeros((8, 32), dtype=torch.uint8, device="cuda")
    s = torch.zeros((8, 1), dtype=torch.float16, device="cuda")
    y = lb.linear(x, w, s, s, None, 4, 64)
    assert y.shape == (0, 8)
    x1 = torch.zeros((1, 64), dtype=torch.bfloat16, device="cuda")
    w0 = torch.zeros((0, 32), dtype=torch.uint8, device="cuda")
    s0 = torch.zeros((0, 1), dtype=torch.float16, device="cuda")
    assert lb.linear(x1, w0, s0, s0, None, 4, 64).shape == (1, 0)


def test_misaligned_pointer_is_rejected_on_gpu():
    L = synth.make_layer(40, 1, 64, 8, 4, 32)
    d = DeviceLayer(L)
    xbig = torch.zeros(64 + 1, dtype=torch.bfloat16, device="cuda")
    xs = xbig[1:].view(1, 64)       # 2-byte offset: not 16-byte aligned
    with pytest.raises(lb.LowbitError) as e:
        lb.linear(xs, d.packed, d.scales, d.zeros, None, 4, 32)
    assert e.value.status == 1


def test_repeated_calls_are_deterministic():
    L = synth.make_layer(41, 1, 4096, 4096, 3, 128)
    d = DeviceLayer(L)
    y1 = d.run()
    y2 = d.run()
    assert torch.equal(y1, y2)


# ---------------------------------------------------------------------------
# Full-size Llama-shaped layers: sampled rows against the oracle.
# ---------------------------------------------------------------------------

def _sampled_check(L, rows, path=0, what=""):
    d = DeviceLayer(L)
    y = d.run(path)
    packed_rows = d.packed[torch.from_numpy(rows).cuda()].cpu().numpy()
    # The oracle packs the sampled rows itself; the device packing is checked bit-exact too.
    ref_packed = ORACLE.pack(L.codes[rows], L.bits)
    assert np.array_equal(packed_rows, ref_packed), what
    ref = ORACLE.linear_rows(L.x, ref_packed, L.scales[rows], L.zeros[rows],
                             None if L.bias is None else L.bias[rows], L.K, L.bits, L.group,
                             np.arange(rows.size))
    check_close(y_to_f64(y)[:, rows], ref, what)


def _rows(N, n, seed):
    r = np.random.default_rng(seed)
    return np.unique(np.concatenate([[0, N - 1], r.choice(N, n, replace=False)]))


@pytest.mark.parametrize("bits", range(1, 8))
@pytest.mark.parametrize("name", list(synth.LLAMA_8B))
def test_llama8b_decode_sweep(bits, name):
    K, N = synth.LLAMA_8B[name]
    L = synth.make_layer(0, 1, K, N, bits, 64)
    _sampled_check(L, _rows(N, 48, bits), what=f"8B {name} b={bits}")


@pytest.mark.parametrize("path", PATHS, ids=lambda p: PATH_IDS[p])
@pytest.mark.parametrize("M", [1, 128])
@pytest.mark.parametrize("name", list(synth.LLAMA_8B))
def test_llama8b_int4wo_128(path, M, name):
    # The int4wo-128 configuration (4-bit codes, groups of 128) of every 8B
    # linear, at batch 1 and 128, through both kernels.
    K, N = synth.LLAMA_8B[name]
    L = synth.make_layer(12, M, K, N, 4, 128, bias=False, outliers=(M > 1))
    _sampled_check(L, _rows(N, 24, M + 7), path=path, what=f"int4wo-128 {name} M={M}")


@pytest.mark.parametrize("bits", [2, 3, 4, 6])
@pytest.mark.parametrize("group", [32, 64, 128, 256])
@pytest.mark.parametrize("model,name", [(m, n) for m in ("3B", "1B") for n in synth.LLAMA_3B])
def test_llama3b1b_decode(bits, group, model, name):
    K, N = (synth.LLAMA_3B if model == "3B" else synth.LLAMA_1B)[name]
    L = synth.make_layer(0, 1, K, N, bits, group)
    _sampled_check(L, _rows(N, 24, group), what=f"{model} {name} b={bits} g={group}")


@pytest.mark.parametrize("path", PATHS, ids=lambda p: PATH_IDS[p])
@pytest.mark.parametrize("M", [2, 4, 8, 16, 32])
@pytest.mark.parametrize("name", list(synth.LLAMA_8B))
def test_llama8b_small_batch(path, M, name):
    K, N = synth.LLAMA_8B[name]
    L = synth.make_layer(0, M, K, N, 4, 128, bias=(name == "qkv"))
    _sampled_check(L, _rows(N, 24, M), path=path, what=f"8B {name} M={M}")


@pytest.mark.parametrize("M", [128, 2048])
@pytest.mark.parametrize("bits", [4, 5])
@pytest.mark.parametrize("name", list(synth.LLAMA_8B))
def test_llama8b_batched(M, bits, name):
    K, N = synth.LLAMA_8B[name]
    L = synth.make_layer(0, M, K, N, bits, 128, bias=True, outliers=True)
    _sampled_check(L, _rows(N, 6 if M == 2048 else 16, M + bits), what=f"8B {name} M={M} b={bits}")


@pytest.mark.parametrize("bits", range(1, 8))
def test_qmm_every_bits_full_tiles(bits):
    # Several 128-row tiles, several K stages, M spanning two 128-row x tiles plus a tail.
    L = synth.make_layer(50 + bits, 300, 1024, 384, bits, 64, bias=True, outliers=True)
    d = DeviceLayer(L)
    check_close(y_to_f64(d.run(lb.PATH_QMM)), _oracle_y(L), f"qmm b={bits}")


@pytest.mark.parametrize("M,K,N,bits,group", [
    (128, 128, 130, 4, 128),    # one K step: the second issuing thread has none
    (40, 384, 300, 3, 128),     # three steps: the two issuing threads take 2 and 1
    (128, 1920, 500, 5, 128),   # 15 steps over a cluster of 8: CTAs with one or two steps
    (130, 2304, 250, 2, 256),   # groups spanning two steps, two x tiles, split over a cluster
    (1, 128, 60, 7, 32),        # g < 128: one issuing thread, four segments per step
    (40, 640, 300, 6, 64),      # g < 128: five steps of two segments
])
def test_qmm_issuers_and_step_counts(M, K, N, bits, group):
    # With g >= 128 the K steps alternate between two MMA-issuing threads (with
    # smaller groups one thread issues them all); step counts of one, odd, and
    # split over a cluster cover every way the steps can fall.
    L = synth.make_layer(70 + K + bits, M, K, N, bits, group, bias=True, outliers=M > 1)
    d = DeviceLayer(L)
    check_close(y_to_f64(d.run(lb.PATH_QMM)), _oracle_y(L), f"qmm {(M, K, N, bits, group)}")


@pytest.mark.parametrize("M,name", [(128, "o"), (8, "down"), (128, "gate_up")])
def test_qmm_split_k_is_deterministic(M, name):
    # Small layers split K over a cluster; the partial sums are added in a
    # fixed order, so repeated calls give identical bits.
    K, N = synth.LLAMA_8B[name]
    L = synth.make_layer(42, M, K, N, 4, 128, bias=True)
    d = DeviceLayer(L)
    y1 = d.run(lb.PATH_QMM)
    y2 = d.run(lb.PATH_QMM)
    assert torch.equal(y1, y2)


def test_auto_path_picks_qmm_for_batches():
    assert lb.select_path(128, 4096, 4096, 4, 128) == lb.PATH_QMM
    assert lb.select_path(1, 4096, 4096, 4, 128) == lb.PATH_QMV


def test_no_wait_timed_out():
    # Every bounded wait in the kernels run above completed in time.
    assert lb.wait_timeouts() == 0


def test_second_device_after_first():
    """Kernel attributes (the raised shared-memory limit) and occupancy are per
    device: a first call on device 1 after calls on device 0 must still run
    (both kernels), and agree with device 0 bit for bit."""
    if torch.cuda.device_count() < 2:
        pytest.skip("needs two GPUs")
    L = synth.make_layer(5, 8, 1024, 300, 4, 64, bias=True)
    outs = []
    for dev in (0, 1):
        with torch.cuda.device(dev):
            w = lb.pack_weights(torch.from_numpy(L.codes).cuda(), 4)
            x = torch.from_numpy(L.x.view(np.int16)).view(torch.bfloat16).cuda()
            s = torch.from_numpy(L.scales.view(np.int16)).view(torch.float16).cuda()
            z = torch.from_numpy(L.zeros.view(np.int16)).view(torch.float16).cuda()
            b = torch.from_numpy(L.bias.view(np.int16)).view(torch.float16).cuda()
            outs.append([lb.linear(x, w, s, z, b, 4, 64, path=p).cpu() for p in PATHS])
            torch.cuda.synchronize()
    for a, b in zip(*outs):
        assert torch.equal(a, b)
