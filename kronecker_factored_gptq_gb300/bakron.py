"""Thin ctypes binding over libbakron.so (argument marshalling only).

Every function here checks tensor devices/dtypes/shapes, allocates outputs
and workspaces with PyTorch (device memory and streams are all PyTorch is used
for), and calls the C entry point of the same name; every step of the solver
runs in the library's CUDA kernels.  There is no CPU path: if the library has
not been built, or no CUDA device is present, the first call raises.
"""

import ctypes
import os

_LIB = None
_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libbakron.so")

OK = 0
STATUS = {0: "BAKRON_OK", 1: "BAKRON_ERR_INVALID_ARG", 2: "BAKRON_ERR_NOT_PD",
          3: "BAKRON_ERR_NONFINITE", 4: "BAKRON_ERR_CODE_RANGE", 5: "BAKRON_ERR_TIMEOUT",
          6: "BAKRON_ERR_UNSUPPORTED", 7: "BAKRON_ERR_CUDA"}
INT32_MIN = -(1 << 31)
INT32_MAX = (1 << 31) - 1

EXPORTS = ["bakron_default_opts", "bakron_status_string", "bakron_version", "bakron_kernel_launches",
           "bakron_workspace_size", "bakron_prepare_workspace_size", "bakron_rowscale",
           "bakron_prepare", "bakron_quantize", "bakron_quantize_antidiag",
           "bakron_quantize_noalloc", "bakron_factors_workspace_size", "bakron_factors",
           "bakron_grid_params", "bakron_quantize_grid", "bakron_batch_workspace_size",
           "bakron_quantize_batch", "bakron_schedule_export", "bakron_fma_probe", "bakron_sm_count",
           "bakron_plan_size", "bakron_plan_init"]
FACTORS_KFAC = 0
FACTORS_SHAMPOO = 1


class PhaseTimes(ctypes.Structure):
    _fields_ = [("leaf_ms", ctypes.c_double), ("prop1_ms", ctypes.c_double),
                ("prop2_ms", ctypes.c_double), ("other_ms", ctypes.c_double),
                ("prop_flops", ctypes.c_double), ("leaf_launches", ctypes.c_int64),
                ("prop_launches", ctypes.c_int64), ("other_launches", ctypes.c_int64),
                ("near_ms", ctypes.c_double), ("near_launches", ctypes.c_int64)]

    def as_dict(self):
        return {f: getattr(self, f) for f, _ in self._fields_}


class Opts(ctypes.Structure):
    _fields_ = [("tile", ctypes.c_int), ("leaf_width", ctypes.c_int), ("use_3xtf32", ctypes.c_int),
                ("spin_budget_cycles", ctypes.c_longlong), ("fault_inject", ctypes.c_int),
                ("times", ctypes.POINTER(PhaseTimes)), ("plan", ctypes.c_void_p)]


class Problem(ctypes.Structure):
    _fields_ = [("W", ctypes.c_void_p), ("m", ctypes.c_int64), ("n", ctypes.c_int64),
                ("UA", ctypes.c_void_p), ("UB", ctypes.c_void_p), ("scale", ctypes.c_void_p),
                ("zero", ctypes.c_void_p), ("group", ctypes.c_int64), ("qmin", ctypes.c_int),
                ("qmax", ctypes.c_int), ("V", ctypes.c_void_p), ("codes", ctypes.c_void_p),
                ("status", ctypes.c_int)]


class BakronError(RuntimeError):
    def __init__(self, status, where):
        self.status = status
        msg = lib().bakron_status_string(status).decode()
        super().__init__("%s: %s (%s)" % (where, STATUS.get(status, status), msg))


def lib():
    """Load libbakron.so (raises if it has not been built)."""
    global _LIB
    if _LIB is not None:
        return _LIB
    if not os.path.exists(LIB_PATH):
        raise RuntimeError("libbakron.so is not built (%s); run __graft_entry__.build()" % LIB_PATH)
    L = ctypes.CDLL(LIB_PATH)
    vp, i64, sz = ctypes.c_void_p, ctypes.c_int64, ctypes.c_size_t
    L.bakron_default_opts.argtypes = [ctypes.POINTER(Opts)]
    L.bakron_default_opts.restype = None
    L.bakron_status_string.argtypes = [ctypes.c_int]
    L.bakron_status_string.restype = ctypes.c_char_p
    L.bakron_version.restype = ctypes.c_int
    L.bakron_kernel_launches.restype = ctypes.c_int64
    L.bakron_workspace_size.argtypes = [i64, i64, ctypes.POINTER(Opts), ctypes.POINTER(sz)]
    L.bakron_prepare_workspace_size.argtypes = [i64, i64, ctypes.POINTER(sz)]
    L.bakron_rowscale.argtypes = [vp, i64, i64, ctypes.c_int, vp, vp]
    L.bakron_prepare.argtypes = [vp, i64, ctypes.c_float, vp, i64, ctypes.c_float,
                                 vp, vp, vp, vp, ctypes.POINTER(i64), vp, sz, vp]
    L.bakron_quantize.argtypes = [vp, i64, i64, vp, vp, vp, ctypes.c_int, ctypes.c_int,
                                  vp, vp, vp, ctypes.POINTER(Opts), vp, sz, vp]
    L.bakron_quantize_antidiag.argtypes = [vp, i64, i64, vp, vp, vp, ctypes.c_int, ctypes.c_int,
                                           vp, vp, vp, vp, ctypes.c_float, ctypes.POINTER(i64),
                                           ctypes.POINTER(Opts), vp, sz, vp]
    L.bakron_quantize_noalloc.argtypes = [vp, i64, i64, vp, vp, vp, ctypes.c_int, ctypes.c_int,
                                          vp, vp, vp]
    L.bakron_grid_params.argtypes = [vp, i64, i64, ctypes.c_int, ctypes.c_int, i64, vp, vp,
                                     ctypes.POINTER(ctypes.c_int), ctypes.POINTER(ctypes.c_int), vp]
    L.bakron_quantize_grid.argtypes = [vp, i64, i64, vp, vp, vp, vp, i64, ctypes.c_int, ctypes.c_int,
                                       vp, vp, vp, ctypes.POINTER(Opts), vp, sz, vp]
    L.bakron_batch_workspace_size.argtypes = [ctypes.c_int, ctypes.POINTER(Problem),
                                              ctypes.POINTER(Opts), ctypes.POINTER(sz)]
    L.bakron_quantize_batch.argtypes = [ctypes.c_int, ctypes.POINTER(Problem), ctypes.POINTER(Opts),
                                        vp, sz, vp]
    L.bakron_factors_workspace_size.argtypes = [i64, i64, i64, ctypes.POINTER(sz)]
    L.bakron_factors.argtypes = [vp, i64, i64, vp, i64, ctypes.c_int, vp, vp, vp, sz, vp]
    L.bakron_schedule_export.argtypes = [ctypes.c_int, i64, i64, vp, i64, ctypes.POINTER(i64)]
    L.bakron_fma_probe.argtypes = [vp, i64, ctypes.c_int, vp]
    L.bakron_plan_size.argtypes = [i64, i64, ctypes.POINTER(sz)]
    L.bakron_plan_init.argtypes = [i64, i64, vp, sz, vp]
    L.bakron_sm_count.restype = ctypes.c_int
    for f in ("bakron_schedule_export", "bakron_workspace_size", "bakron_prepare_workspace_size", "bakron_rowscale",
              "bakron_prepare", "bakron_quantize", "bakron_quantize_antidiag",
              "bakron_quantize_noalloc", "bakron_factors_workspace_size", "bakron_factors",
              "bakron_grid_params", "bakron_quantize_grid", "bakron_batch_workspace_size",
              "bakron_quantize_batch", "bakron_fma_probe", "bakron_plan_size",
              "bakron_plan_init"):
        getattr(L, f).restype = ctypes.c_int
    _LIB = L
    return L


def kernel_launches():
    """Kernels the library has launched in this process so far."""
    return int(lib().bakron_kernel_launches())


def sm_count():
    """Streaming multiprocessors of the current CUDA device."""
    return int(lib().bakron_sm_count())


def fma_probe(out, blocks, iters):
    """Enqueue the FP32 FMA throughput probe on the current stream (see
    bakron_fma_probe); ``out`` is a float32 CUDA tensor of blocks * 256
    elements.  Returns the flops it performs."""
    import torch
    assert out.dtype == torch.float32 and out.is_cuda and out.numel() >= blocks * 256
    st = lib().bakron_fma_probe(ctypes.c_void_p(out.data_ptr()), int(blocks), int(iters),
                                ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    if st != OK:
        raise BakronError(st, "bakron_fma_probe")
    return 2.0 * blocks * 256 * iters * 128


SCHEDULE_SOLVE = 0
SCHEDULE_ROWS = 1
SCHEDULE_PREPARE = 2


def schedule_export(kind, M, N=1):
    """The library's work lists for a shape in 128-tiles (host only, no GPU):
    an int32 numpy array in the layout bakron_schedule_export documents."""
    import numpy as np
    n = ctypes.c_int64(0)
    st = lib().bakron_schedule_export(int(kind), int(M), int(N), None, 0, ctypes.byref(n))
    if st != OK:
        raise BakronError(st, "bakron_schedule_export")
    out = np.zeros(max(1, n.value), dtype=np.int32)
    st = lib().bakron_schedule_export(int(kind), int(M), int(N), ctypes.c_void_p(out.ctypes.data),
                                      n.value, ctypes.byref(n))
    if st != OK:
        raise BakronError(st, "bakron_schedule_export")
    return out[:n.value]


def default_opts(**kw):
    o = Opts()
    lib().bakron_default_opts(ctypes.byref(o))
    for k, v in kw.items():
        setattr(o, k, v)
    return o


def _check(st, where):
    if st != OK:
        raise BakronError(st, where)


def _torch():
    import torch
    if not torch.cuda.is_available():
        raise RuntimeError("no CUDA device: the BaKron library runs on the GPU only")
    return torch


def _dev(t, dtype, shape, name):
    torch = _torch()
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise ValueError("%s must be a CUDA tensor" % name)
    if t.dtype != dtype:
        raise ValueError("%s must be %s, got %s" % (name, dtype, t.dtype))
    if tuple(t.shape) != tuple(shape):
        raise ValueError("%s must have shape %s, got %s" % (name, tuple(shape), tuple(t.shape)))
    if not t.is_contiguous():
        raise ValueError("%s must be contiguous" % name)
    return ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    torch = _torch()
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def workspace_size(m, n, opts=None):
    b = ctypes.c_size_t(0)
    _check(lib().bakron_workspace_size(m, n, ctypes.byref(opts) if opts else None, ctypes.byref(b)),
           "bakron_workspace_size")
    return b.value


def plan_size(m, n):
    b = ctypes.c_size_t(0)
    _check(lib().bakron_plan_size(m, n, ctypes.byref(b)), "bakron_plan_size")
    return b.value


def bakron_plan_init(m, n, plan=None, stream=None):
    """The work-list plan of the m x n shape in a device buffer (uint8 tensor,
    allocated here when ``plan`` is None); pass it as ``opts.plan``."""
    torch = _torch()
    nb = plan_size(m, n)
    if plan is None:
        plan = torch.empty(nb, dtype=torch.uint8, device="cuda")
    elif plan.numel() * plan.element_size() < nb:
        raise ValueError("plan buffer too small: need %d bytes" % nb)
    _check(lib().bakron_plan_init(m, n, ctypes.c_void_p(plan.data_ptr()), nb, _stream(stream)),
           "bakron_plan_init")
    return plan


def prepare_workspace_size(n, m):
    b = ctypes.c_size_t(0)
    _check(lib().bakron_prepare_workspace_size(n, m, ctypes.byref(b)), "bakron_prepare_workspace_size")
    return b.value


def _ws(nbytes, workspace):
    torch = _torch()
    if workspace is not None:
        if workspace.numel() * workspace.element_size() < nbytes:
            raise ValueError("workspace too small: need %d bytes" % nbytes)
        return workspace
    return torch.empty(nbytes, dtype=torch.uint8, device="cuda")


def bakron_rowscale(W, qmax, out=None, stream=None):
    torch = _torch()
    m, n = W.shape
    if out is None:
        out = torch.empty(m, dtype=torch.float32, device=W.device)
    _check(lib().bakron_rowscale(_dev(W, torch.float32, (m, n), "W"), m, n, int(qmax),
                                 _dev(out, torch.float32, (m,), "scale"), _stream(stream)),
           "bakron_rowscale")
    return out


def bakron_prepare(A, damp_A, B=None, damp_B=0.0, want_L=False, workspace=None, stream=None,
                   out=None):
    """Returns (UA, UB, LA, LB, info); UB/LB are None when B is None."""
    torch = _torch()
    n = A.shape[0]
    m = 0 if B is None else B.shape[0]
    if out is not None:
        UA, UB = out
    else:
        UA = torch.empty((n, n), dtype=torch.float32, device=A.device)
        UB = None if B is None else torch.empty((m, m), dtype=torch.float32, device=A.device)
    LA = torch.empty_like(UA) if want_L else None
    LB = torch.empty_like(UB) if (want_L and B is not None) else None
    nb = prepare_workspace_size(n, m)
    ws = _ws(nb, workspace)
    info = (ctypes.c_int64 * 2)(-1, -1)
    st = lib().bakron_prepare(
        _dev(A, torch.float32, (n, n), "A"), n, float(damp_A),
        None if B is None else _dev(B, torch.float32, (m, m), "B"), m, float(damp_B),
        _dev(UA, torch.float32, (n, n), "UA"),
        None if UB is None else _dev(UB, torch.float32, (m, m), "UB"),
        None if LA is None else _dev(LA, torch.float32, (n, n), "LA"),
        None if LB is None else _dev(LB, torch.float32, (m, m), "LB"),
        info, ctypes.c_void_p(ws.data_ptr()), nb, _stream(stream))
    if st != OK:
        err = BakronError(st, "bakron_prepare")
        err.info = (info[0], info[1])
        raise err
    return UA, UB, LA, LB, (info[0], info[1])


def bakron_quantize(W, UA, UB, scale, qmin, qmax, want_preround=False, opts=None, workspace=None,
                    stream=None, out=None):
    """Returns (V, codes, preround-or-None).  UB=None means B = I: one-sided
    GPTQ with Hessian A for every row, solved by the library's row path."""
    torch = _torch()
    m, n = W.shape
    if out is None:
        V = torch.empty((m, n), dtype=torch.float32, device=W.device)
        codes = torch.empty((m, n), dtype=torch.int8, device=W.device)
    else:
        V, codes = out
    pre = torch.empty((m, n), dtype=torch.float32, device=W.device) if want_preround else None
    nb = workspace_size(m, n, opts)
    ws = _ws(nb, workspace)
    st = lib().bakron_quantize(
        _dev(W, torch.float32, (m, n), "W"), m, n,
        _dev(UA, torch.float32, (n, n), "UA"),
        None if UB is None else _dev(UB, torch.float32, (m, m), "UB"),
        _dev(scale, torch.float32, (m,), "scale"), int(qmin), int(qmax),
        _dev(V, torch.float32, (m, n), "V"), _dev(codes, torch.int8, (m, n), "codes"),
        None if pre is None else _dev(pre, torch.float32, (m, n), "preround"),
        ctypes.byref(opts) if opts is not None else None,
        ctypes.c_void_p(ws.data_ptr()), nb, _stream(stream))
    _check(st, "bakron_quantize")
    return V, codes, pre


def grid_groups(n, group):
    """Number of column groups of a grid (group 0/None or >= n: one per row)."""
    if not group or group >= n:
        return 1
    if group % 32:
        raise ValueError("group must be a multiple of 32 (or cover the whole row)")
    return -(-n // group)


def bakron_grid_params(W, bits, asymmetric=False, group=None, stream=None):
    """Grid of a b-bit base quantizer on the original W: returns
    (scale, zero, qmin, qmax) with scale/zero of shape (m, groups)."""
    torch = _torch()
    m, n = W.shape
    ng = grid_groups(n, group)
    scale = torch.empty((m, ng), dtype=torch.float32, device=W.device)
    zero = torch.empty((m, ng), dtype=torch.float32, device=W.device)
    qmin, qmax = ctypes.c_int(0), ctypes.c_int(0)
    st = lib().bakron_grid_params(_dev(W, torch.float32, (m, n), "W"), m, n, int(bits),
                                  1 if asymmetric else 0, int(group or 0),
                                  ctypes.c_void_p(scale.data_ptr()), ctypes.c_void_p(zero.data_ptr()),
                                  ctypes.byref(qmin), ctypes.byref(qmax), _stream(stream))
    _check(st, "bakron_grid_params")
    return scale, zero, qmin.value, qmax.value


def bakron_quantize_grid(W, UA, UB, scale, zero, group, qmin, qmax, want_preround=False, opts=None,
                         workspace=None, stream=None, out=None):
    """bakron_quantize on a grid (scale/zero of shape (m, groups)); UB=None
    means B = I.  Returns (V, codes, preround-or-None)."""
    torch = _torch()
    m, n = W.shape
    ng = grid_groups(n, group)
    if out is None:
        V = torch.empty((m, n), dtype=torch.float32, device=W.device)
        codes = torch.empty((m, n), dtype=torch.int8, device=W.device)
    else:
        V, codes = out
    pre = torch.empty((m, n), dtype=torch.float32, device=W.device) if want_preround else None
    nb = workspace_size(m, n, opts)
    ws = _ws(nb, workspace)
    st = lib().bakron_quantize_grid(
        _dev(W, torch.float32, (m, n), "W"), m, n, _dev(UA, torch.float32, (n, n), "UA"),
        None if UB is None else _dev(UB, torch.float32, (m, m), "UB"),
        _dev(scale, torch.float32, (m, ng), "scale"),
        None if zero is None else _dev(zero, torch.float32, (m, ng), "zero"),
        int(group or 0), int(qmin), int(qmax),
        _dev(V, torch.float32, (m, n), "V"), _dev(codes, torch.int8, (m, n), "codes"),
        None if pre is None else _dev(pre, torch.float32, (m, n), "preround"),
        ctypes.byref(opts) if opts is not None else None,
        ctypes.c_void_p(ws.data_ptr()), nb, _stream(stream))
    _check(st, "bakron_quantize_grid")
    return V, codes, pre


def bakron_quantize_batch(problems, opts=None, workspace=None, stream=None, outs=None):
    """Several independent solves at once.  ``problems``: sequence of dicts
    with W, UA, UB (None = B = I), scale, zero (None = 0), group (None = per
    row), qmin, qmax.  Returns a list of (V, codes); raises BakronError with
    ``statuses`` (one per problem) if any problem failed."""
    torch = _torch()
    arr = (Problem * len(problems))()
    keep = []
    for k, pr in enumerate(problems):
        W = pr["W"]
        m, n = W.shape
        ng = grid_groups(n, pr.get("group"))
        if outs is None:
            V = torch.empty((m, n), dtype=torch.float32, device=W.device)
            C = torch.empty((m, n), dtype=torch.int8, device=W.device)
        else:
            V, C = outs[k]
        UB, zero = pr.get("UB"), pr.get("zero")
        arr[k] = Problem(
            _dev(W, torch.float32, (m, n), "W"), m, n, _dev(pr["UA"], torch.float32, (n, n), "UA"),
            None if UB is None else _dev(UB, torch.float32, (m, m), "UB"),
            _dev(pr["scale"], torch.float32, (m, ng) if ng > 1 or pr["scale"].dim() == 2 else (m,),
                 "scale"),
            None if zero is None else _dev(zero, torch.float32, (m, ng), "zero"),
            int(pr.get("group") or 0), int(pr["qmin"]), int(pr["qmax"]),
            _dev(V, torch.float32, (m, n), "V"), _dev(C, torch.int8, (m, n), "codes"), 0)
        keep.append((V, C))
    size = ctypes.c_size_t(0)
    o = ctypes.byref(opts) if opts is not None else None
    _check(lib().bakron_batch_workspace_size(len(problems), arr, o, ctypes.byref(size)),
           "bakron_batch_workspace_size")
    ws = _ws(size.value, workspace)
    st = lib().bakron_quantize_batch(len(problems), arr, o, ctypes.c_void_p(ws.data_ptr()),
                                     size.value, _stream(stream))
    if st != OK:
        err = BakronError(st, "bakron_quantize_batch")
        err.statuses = [arr[k].status for k in range(len(problems))]
        raise err
    return keep


def bakron_quantize_antidiag(W, UA, UB, scale, qmin, qmax, guide_codes=None, guide_tol=1e-4,
                             want_preround=False, opts=None, workspace=None, stream=None):
    """Returns (V, codes, preround-or-None, overrides)."""
    torch = _torch()
    m, n = W.shape
    V = torch.empty((m, n), dtype=torch.float32, device=W.device)
    codes = torch.empty((m, n), dtype=torch.int8, device=W.device)
    pre = torch.empty((m, n), dtype=torch.float32, device=W.device) if want_preround else None
    nb = workspace_size(m, n, opts)
    ws = _ws(nb, workspace)
    over = ctypes.c_int64(0)
    st = lib().bakron_quantize_antidiag(
        _dev(W, torch.float32, (m, n), "W"), m, n,
        _dev(UA, torch.float32, (n, n), "UA"), _dev(UB, torch.float32, (m, m), "UB"),
        _dev(scale, torch.float32, (m,), "scale"), int(qmin), int(qmax),
        _dev(V, torch.float32, (m, n), "V"), _dev(codes, torch.int8, (m, n), "codes"),
        None if pre is None else _dev(pre, torch.float32, (m, n), "preround"),
        None if guide_codes is None else _dev(guide_codes, torch.int8, (m, n), "guide_codes"),
        float(guide_tol), ctypes.byref(over),
        ctypes.byref(opts) if opts is not None else None,
        ctypes.c_void_p(ws.data_ptr()), nb, _stream(stream))
    _check(st, "bakron_quantize_antidiag")
    return V, codes, pre, over.value


NOALLOC_MAX_DIM = 512


def bakron_quantize_noalloc(W, UA, UB, scale, qmin, qmax, out=None, stream=None):
    """bakron_quantize without a workspace (the library's fixed scratch array;
    m, n <= 512).  For callers that cannot allocate device memory, pass
    pre-allocated ``out=(V, codes)``; this wrapper then allocates nothing
    either.  Returns (V, codes)."""
    torch = _torch()
    m, n = W.shape
    if out is None:
        V = torch.empty((m, n), dtype=torch.float32, device=W.device)
        codes = torch.empty((m, n), dtype=torch.int8, device=W.device)
    else:
        V, codes = out
    st = lib().bakron_quantize_noalloc(
        _dev(W, torch.float32, (m, n), "W"), m, n,
        _dev(UA, torch.float32, (n, n), "UA"), _dev(UB, torch.float32, (m, m), "UB"),
        _dev(scale, torch.float32, (m,), "scale"), int(qmin), int(qmax),
        _dev(V, torch.float32, (m, n), "V"), _dev(codes, torch.int8, (m, n), "codes"),
        _stream(stream))
    _check(st, "bakron_quantize_noalloc")
    return V, codes


def factors_workspace_size(N, n, m):
    size = ctypes.c_size_t(0)
    _check(lib().bakron_factors_workspace_size(N, n, m, ctypes.byref(size)),
           "bakron_factors_workspace_size")
    return size.value


def bakron_factors(X=None, G=None, mode=FACTORS_KFAC, want_A=True, want_B=True, workspace=None,
                   stream=None):
    """Kronecker factors (A, B) from samples: rows of X (N x n) are input
    activations, rows of G (N x m) output gradients.  mode FACTORS_KFAC or
    FACTORS_SHAMPOO; an unwanted factor comes back as None."""
    torch = _torch()
    ref = X if X is not None else G
    N = ref.shape[0]
    n = 0 if X is None else X.shape[1]
    m = 0 if G is None else G.shape[1]
    A = torch.empty((n, n), dtype=torch.float32, device=ref.device) if (want_A and X is not None) else None
    B = torch.empty((m, m), dtype=torch.float32, device=ref.device) if (want_B and G is not None) else None
    size = ctypes.c_size_t(0)
    _check(lib().bakron_factors_workspace_size(N, n, m, ctypes.byref(size)),
           "bakron_factors_workspace_size")
    ws = _ws(size.value, workspace)
    st = lib().bakron_factors(
        None if X is None else _dev(X, torch.float32, (N, n), "X"), N, n,
        None if G is None else _dev(G, torch.float32, (N, m), "G"), m, int(mode),
        None if A is None else _dev(A, torch.float32, (n, n), "A"),
        None if B is None else _dev(B, torch.float32, (m, m), "B"),
        ctypes.c_void_p(ws.data_ptr()), size.value, _stream(stream))
    _check(st, "bakron_factors")
    return A, B


class Solver:
    """The whole path on one GPU: row grid, factor preparation, solve.

    Workspaces, the shape's work-list plan and the outputs are allocated once
    per shape and reused, so repeated solves of one shape allocate nothing.
    """

    def __init__(self, m, n, bits=None, qmin=None, qmax=None, opts=None, stream=None):
        torch = _torch()
        self.m, self.n = m, n
        if bits is not None:
            self.qmax = (1 << (bits - 1)) - 1
            self.qmin = -(self.qmax + 1)
        else:
            self.qmin, self.qmax = qmin, qmax
        self.opts = opts if opts is not None else default_opts()
        self.stream = stream
        dev = "cuda"
        self.plan = bakron_plan_init(m, n, stream=stream)
        self.ws_q = torch.empty(workspace_size(m, n, opts), dtype=torch.uint8, device=dev)
        self.ws_p = torch.empty(prepare_workspace_size(n, m), dtype=torch.uint8, device=dev)
        self.scale = torch.empty(m, dtype=torch.float32, device=dev)
        self.UA = torch.empty((n, n), dtype=torch.float32, device=dev)
        self.UB = torch.empty((m, m), dtype=torch.float32, device=dev)
        self.V = torch.empty((m, n), dtype=torch.float32, device=dev)
        self.codes = torch.empty((m, n), dtype=torch.int8, device=dev)

    def rowscale(self, W):
        return bakron_rowscale(W, self.qmax, out=self.scale, stream=self.stream)

    def prepare(self, A, damp_A, B, damp_B):
        bakron_prepare(A, damp_A, B, damp_B, workspace=self.ws_p, stream=self.stream,
                       out=(self.UA, self.UB))
        return self.UA, self.UB

    def quantize(self, W, UA=None, UB=None, scale=None, want_preround=False):
        if self.opts is not None and not self.opts.plan:
            self.opts.plan = self.plan.data_ptr()
        return bakron_quantize(W, self.UA if UA is None else UA, self.UB if UB is None else UB,
                               self.scale if scale is None else scale, self.qmin, self.qmax,
                               want_preround=want_preround, opts=self.opts, workspace=self.ws_q,
                               stream=self.stream, out=(self.V, self.codes))

    def solve(self, W, A, damp_A, B, damp_B):
        """Row grid + factor preparation + BaKron solve; returns (V, codes)."""
        self.rowscale(W)
        self.prepare(A, damp_A, B, damp_B)
        return self.quantize(W)[:2]
