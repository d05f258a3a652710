"""Host-side contract checks of the C ABI, run in a subprocess with no visible
CUDA device (CUDA_VISIBLE_DEVICES="").

Every case calls an entry point with placeholder (never dereferenced) device
addresses and checks the status the validation layer returns.  Because no
device is visible, a case that wrongly passed validation would fail in the
device query (EP_ERR_CUDA) instead of launching anything.

Run as a script: exits 0 if every case returns its expected status, 1
otherwise (printing the mismatches).
"""
import ctypes
import json
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

F32, F16, BF16, F64 = 0, 1, 2, 7
OK, INVALID, UNSUPPORTED, WORKSPACE, CUDA = 0, 1, 2, 3, 4

# placeholder device addresses: distinct, far apart, 256-byte aligned
A, B, C, D, E, F, G = (0x7F0000000000 + i * (1 << 32) for i in range(7))


def shp(*d):
    return (ctypes.c_int64 * max(1, len(d)))(*d), len(d)


def sln(lib, t=F32, inp=A, in_shape=(4, 8), skip=B, skip_shape=(4, 8), gamma=C, beta=D, bias=E, eps=1e-12,
        out=F, res=None):
    s_in, r_in = shp(*in_shape)
    s_sk, r_sk = shp(*skip_shape)
    return lib.ep_skip_layer_norm(t, inp, s_in, r_in, skip, s_sk, r_sk, gamma, beta, bias, eps, out, res, None)


def sln_ex(lib, t=F32, inp=A, in_shape=(4, 8), skip=B, skip_shape=(4, 8), gamma=C, beta=D, bias=E, eps=1e-12,
           simplified=0, out=F, res=None, mean=None, inv=None):
    s_in, r_in = shp(*in_shape)
    s_sk, r_sk = shp(*skip_shape)
    return lib.ep_skip_layer_norm_ex(t, inp, s_in, r_in, skip, s_sk, r_sk, gamma, beta, bias, eps, simplified,
                                     out, res, mean, inv, None)


def softmax(lib, t=F32, data=A, shape=(4, 8), bias=B, bias_numel=8, axis=1, inner=1, out=C, ws=None, wsb=0):
    s, r = shp(*shape)
    return lib.ep_bias_softmax(t, data, s, r, bias, bias_numel, axis, inner, out, ws, wsb, None)


def softmax_noalloc(lib, t=F32, data=A, shape=(4, 8), bias=B, bias_numel=8, axis=1, inner=1, out=C):
    s, r = shp(*shape)
    return lib.ep_bias_softmax_noalloc(t, data, s, r, bias, bias_numel, axis, inner, out, None)


def bias_add(lib, t=F16, x=A, shape=(2, 3, 8), bias=B, skip=C, y=D):
    s, _ = shp(*shape)
    return lib.ep_bias_add(t, x, s, bias, skip, y, None)


def gelu(lib, t=F16, x=A, n=100, alpha=1.702, y=B):
    return lib.ep_quick_gelu(t, x, n, alpha, y, None)


def cases(lib):
    es32 = 4
    n48 = 4 * 8 * es32  # bytes of a (4, 8) f32 tensor
    return [
        # --- SkipLayerNormalization: dtype / rank
        ("sln bf16 ok", sln(lib, t=BF16), CUDA),
        ("sln f64 unsupported", sln(lib, t=F64), UNSUPPORTED),
        ("sln rank 1 unsupported", sln(lib, in_shape=(8,), skip_shape=(8,)), UNSUPPORTED),
        ("sln rank 4 unsupported", sln(lib, in_shape=(1, 2, 4, 8), skip_shape=(1, 2, 4, 8)), UNSUPPORTED),
        # --- hidden size, skip shapes, epsilon
        ("sln H = 0", sln(lib, in_shape=(4, 0), skip_shape=(4, 0)), INVALID),
        ("sln negative dim", sln(lib, in_shape=(-4, 8), skip_shape=(-4, 8)), INVALID),
        ("sln rank-2 skip must match", sln(lib, in_shape=(4, 8), skip_shape=(2, 8)), INVALID),
        ("sln rank-2 skip (1,H) rejected", sln(lib, in_shape=(4, 8), skip_shape=(1, 8)), INVALID),
        ("sln rank-3 skip (1,S,H) ok", sln(lib, in_shape=(2, 3, 8), skip_shape=(1, 3, 8)), CUDA),
        ("sln rank-3 skip (S,H) ok", sln(lib, in_shape=(2, 3, 8), skip_shape=(3, 8)), CUDA),
        ("sln rank-3 skip exact ok", sln(lib, in_shape=(2, 3, 8), skip_shape=(2, 3, 8)), CUDA),
        ("sln rank-3 skip (2,1,8) rejected", sln(lib, in_shape=(2, 3, 8), skip_shape=(2, 1, 8)), INVALID),
        ("sln rank-3 skip (1,8) rejected", sln(lib, in_shape=(2, 3, 8), skip_shape=(1, 8)), INVALID),
        ("sln rank-3 skip (3,4) rejected", sln(lib, in_shape=(2, 3, 8), skip_shape=(3, 4)), INVALID),
        ("sln negative epsilon", sln(lib, eps=-1e-5), INVALID),
        ("sln NaN epsilon", sln(lib, eps=float("nan")), INVALID),
        ("sln epsilon 0 ok", sln(lib, eps=0.0), CUDA),
        # --- required pointers, alignment, empties
        ("sln NULL input", sln(lib, inp=None), INVALID),
        ("sln NULL gamma", sln(lib, gamma=None), INVALID),
        ("sln NULL output", sln(lib, out=None), INVALID),
        ("sln NULL beta/bias ok", sln(lib, beta=None, bias=None), CUDA),
        ("sln misaligned f32 pointer", sln(lib, inp=A + 2), INVALID),
        ("sln misaligned f16 pointer", sln(lib, t=F16, gamma=C + 1), INVALID),
        ("sln f16 2-byte offset ok", sln(lib, t=F16, inp=A + 2), CUDA),
        ("sln empty rows launch nothing", sln(lib, inp=None, skip=None, gamma=None, out=None,
                                              in_shape=(0, 3, 8), skip_shape=(0, 3, 8)), OK),
        # --- overlaps
        ("sln output == input (in place) ok", sln(lib, out=A), CUDA),
        ("sln output partially overlaps input", sln(lib, out=A + 16), INVALID),
        ("sln output overlaps gamma", sln(lib, out=C), INVALID),
        ("sln sum == skip (in place) ok", sln(lib, res=B), CUDA),
        ("sln sum overlaps output", sln(lib, res=F + 8), INVALID),
        ("sln output aliases broadcast skip", sln(lib, in_shape=(2, 3, 8), skip_shape=(3, 8), out=B), INVALID),
        ("sln output right after input ok", sln(lib, out=A + n48), CUDA),
        # --- SkipLayerNormalization, RMS form and statistics
        ("sln_ex simplified ok", sln_ex(lib, simplified=1, beta=None), CUDA),
        ("sln_ex simplified must be 0/1", sln_ex(lib, simplified=2), INVALID),
        ("sln_ex statistics ok", sln_ex(lib, mean=G, inv=G + 4096), CUDA),
        ("sln_ex misaligned mean", sln_ex(lib, mean=G + 2), INVALID),
        ("sln_ex mean overlaps inv_std_dev", sln_ex(lib, mean=G, inv=G + 8), INVALID),
        ("sln_ex mean overlaps output", sln_ex(lib, mean=F + 4), INVALID),
        ("sln_ex inv_std_dev overlaps input", sln_ex(lib, inv=A), INVALID),
        ("sln_ex f64 unsupported", sln_ex(lib, t=F64), UNSUPPORTED),
        # --- BiasSoftmax
        ("softmax bf16 ok", softmax(lib, t=BF16), CUDA),
        ("softmax f64 unsupported", softmax(lib, t=F64), UNSUPPORTED),
        ("softmax rank 0", softmax(lib, shape=()), INVALID),
        ("softmax rank 17 unsupported", softmax(lib, shape=(1,) * 17, bias_numel=1, axis=16), UNSUPPORTED),
        ("softmax axis = rank", softmax(lib, axis=2), INVALID),
        ("softmax axis = -rank ok", softmax(lib, axis=-2, bias_numel=32), CUDA),
        ("softmax axis < -rank", softmax(lib, axis=-3), INVALID),
        ("softmax bias not whole rows", softmax(lib, bias_numel=12), INVALID),
        ("softmax bias rows do not divide", softmax(lib, shape=(6, 8), bias_numel=32), INVALID),
        ("softmax more bias rows than data rows", softmax(lib, bias_numel=40), INVALID),
        ("softmax empty bias, data not empty", softmax(lib, bias_numel=0), INVALID),
        ("softmax both empty ok", softmax(lib, shape=(0, 8), bias_numel=0, data=None, bias=None, out=None), OK),
        ("softmax blockSize 0 with bias", softmax(lib, shape=(4, 0), bias_numel=4), INVALID),
        ("softmax negative bias numel", softmax(lib, bias_numel=-8), INVALID),
        ("softmax NULL bias", softmax(lib, bias=None), INVALID),
        ("softmax misaligned", softmax(lib, t=F32, data=A + 2), INVALID),
        ("softmax in place ok", softmax(lib, out=A), CUDA),
        ("softmax output overlaps bias", softmax(lib, out=B + 4), INVALID),
        ("softmax inner flag any nonzero ok", softmax(lib, inner=7), CUDA),
        ("softmax long row without workspace", softmax(lib, shape=(2, 70000), bias_numel=70000), WORKSPACE),
        ("softmax long row, small workspace", softmax(lib, shape=(2, 70000), bias_numel=70000, ws=D, wsb=8), WORKSPACE),
        ("softmax long row, misaligned workspace",
         softmax(lib, shape=(2, 70000), bias_numel=70000, ws=D + 8, wsb=1 << 20), WORKSPACE),
        ("softmax long row, workspace ok",
         softmax(lib, shape=(2, 70000), bias_numel=70000, ws=D, wsb=1 << 20), CUDA),
        ("softmax long row, workspace overlaps data",
         softmax(lib, shape=(2, 70000), bias_numel=70000, ws=A, wsb=1 << 20), WORKSPACE),
        # --- BiasSoftmax without a workspace (fixed scratch of 131072 chunk entries)
        ("softmax noalloc one chunk beyond the fixed scratch",      # f32: 26215 rows x 5 chunks = 131075
         softmax_noalloc(lib, shape=(26215, 16385), bias_numel=16385), WORKSPACE),
        ("softmax noalloc just within the fixed scratch",           # 26214 x 5 = 131070
         softmax_noalloc(lib, shape=(26214, 16385), bias_numel=16385), CUDA),
        ("softmax noalloc f16 within the fixed scratch",            # f16: 43690 rows x 3 chunks
         softmax_noalloc(lib, t=F16, shape=(43690, 16385), bias_numel=16385), CUDA),
        ("softmax noalloc f16 beyond the fixed scratch",            # 43691 x 3 = 131073
         softmax_noalloc(lib, t=F16, shape=(43691, 16385), bias_numel=16385), WORKSPACE),
        ("softmax noalloc long rows within the limit", softmax_noalloc(lib, shape=(2, 70000), bias_numel=70000), CUDA),
        ("softmax noalloc row path, any row count", softmax_noalloc(lib, shape=(1 << 22, 512), bias_numel=512), CUDA),
        ("softmax noalloc contract", softmax_noalloc(lib, bias_numel=12), INVALID),
        ("softmax noalloc in place ok", softmax_noalloc(lib, out=A), CUDA),
        ("softmax noalloc empty ok", softmax_noalloc(lib, shape=(0, 8), bias_numel=0, data=None, bias=None, out=None), OK),
        # --- failure detection
        ("selftest limit 0", lib.ep_selftest_bounded_wait(0, ctypes.byref(ctypes.c_uint64()), None), INVALID),
        ("selftest limit above 1 s", lib.ep_selftest_bounded_wait(1000001, ctypes.byref(ctypes.c_uint64()), None), INVALID),
        ("selftest NULL result", lib.ep_selftest_bounded_wait(1000, None, None), INVALID),
        ("selftest valid (no device)", lib.ep_selftest_bounded_wait(1000, ctypes.byref(ctypes.c_uint64()), None), CUDA),
        ("pipeline_timeouts NULL", lib.ep_pipeline_timeouts(None, 0), INVALID),
        ("pipeline_timeouts valid (no device)", lib.ep_pipeline_timeouts(ctypes.byref(ctypes.c_uint64()), 0), CUDA),
        # --- BiasAdd
        ("bias_add bf16 ok", bias_add(lib, t=BF16), CUDA),
        ("bias_add f64 unsupported", bias_add(lib, t=F64), UNSUPPORTED),
        ("bias_add negative dim", bias_add(lib, shape=(2, -3, 8)), INVALID),
        ("bias_add empty ok", bias_add(lib, shape=(0, 3, 8), x=None, bias=None, skip=None, y=None), OK),
        ("bias_add NULL skip", bias_add(lib, skip=None), INVALID),
        ("bias_add misaligned", bias_add(lib, y=D + 1), INVALID),
        ("bias_add in place on X ok", bias_add(lib, y=A), CUDA),
        ("bias_add in place on skip ok", bias_add(lib, y=C), CUDA),
        ("bias_add Y overlaps bias", bias_add(lib, y=B), INVALID),
        ("bias_add Y partially overlaps X", bias_add(lib, y=A + 2), INVALID),
        # --- QuickGelu
        ("gelu bf16 ok", gelu(lib, t=BF16), CUDA),
        ("gelu f64 unsupported", gelu(lib, t=F64), UNSUPPORTED),
        ("gelu negative numel", gelu(lib, n=-1), INVALID),
        ("gelu empty ok", gelu(lib, n=0, x=None, y=None), OK),
        ("gelu NULL X", gelu(lib, x=None), INVALID),
        ("gelu misaligned", gelu(lib, t=F32, x=A + 2), INVALID),
        ("gelu in place ok", gelu(lib, y=A), CUDA),
        ("gelu partial overlap", gelu(lib, y=A + 2), INVALID),
        ("gelu NaN alpha accepted", gelu(lib, alpha=float("nan")), CUDA),
    ]


def main():
    assert os.environ.get("CUDA_VISIBLE_DEVICES", None) == "", "run with CUDA_VISIBLE_DEVICES=''"
    from transformer_epilogue_gb300 import _binding
    lib = _binding.load_library()
    bad = []
    n0 = lib.ep_kernel_launch_count()
    for name, got, want in cases(lib):
        msg = lib.ep_last_error().decode()
        if got != want:
            bad.append((name, got, want, msg))
        if got != OK and not msg:
            bad.append((name, got, want, "empty error message"))
    # workspace size queries are pure host arithmetic
    s, r = shp(2, 70000)
    ws = lib.ep_bias_softmax_workspace_size(F32, s, r, 1)
    if ws != 2 * 18 * 8:         # f32: ceil(70000 / 4096) = 18 chunks of (max, sum) floats per row
        bad.append(("workspace size (2, 70000)", ws, 288, ""))
    if lib.ep_bias_softmax_workspace_size(F16, s, r, 1) != 2 * 9 * 8:   # f16: 8192-column chunks
        bad.append(("workspace size f16 (2, 70000)", lib.ep_bias_softmax_workspace_size(F16, s, r, 1), 144, ""))
    s, r = shp(262144, 512)
    if lib.ep_bias_softmax_workspace_size(F16, s, r, 1) != 0:
        bad.append(("workspace size of a row-path shape", 1, 0, ""))
    if lib.ep_bias_softmax_workspace_size(F64, s, r, 1) != 0:
        bad.append(("workspace size of an unsupported dtype", 1, 0, ""))
    s2, r2 = shp(2, 70000)
    if lib.ep_bias_softmax_workspace_size(BF16, s2, r2, 1) != 2 * 9 * 8:   # bf16: 8192-column chunks
        bad.append(("workspace size bf16 (2, 70000)", lib.ep_bias_softmax_workspace_size(BF16, s2, r2, 1), 144, ""))
    if lib.ep_kernel_launch_count() != n0:
        bad.append(("launch count moved", lib.ep_kernel_launch_count(), n0, ""))
    if lib.ep_abi_version() != 1:
        bad.append(("abi version", lib.ep_abi_version(), 1, ""))
    for code, name in [(0, "EP_OK"), (1, "EP_ERR_INVALID_ARG"), (2, "EP_ERR_UNSUPPORTED"), (3, "EP_ERR_WORKSPACE"),
                       (4, "EP_ERR_CUDA")]:
        if lib.ep_status_name(code).decode() != name:
            bad.append(("status name", code, name, ""))
    print(json.dumps({"cases": len(cases(lib)), "failures": bad}))
    return 1 if bad else 0


if __name__ == "__main__":
    sys.exit(main())
