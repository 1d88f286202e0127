"""MFA decode attention for GB300 (sm_103a).

Thin ctypes binding over ``libmfa.so`` (CUDA kernels + C ABI, see include/mfa.h).
Every step of the decode runs in the library's kernels; this module only
marshals arguments.  PyTorch supplies device memory and the current stream.

The operation is Step-3's MFA decode step (paperlayer.ai/abs/2507.19427v1,
section 2 "Step-3 Model Card" and section 5 "Model-System Co-design"): 64 query
heads of width 256 over one shared K head and one shared V head held in a paged
KV cache of 64-token pages, out = softmax(q K^T * scale) V and its log-sum-exp.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional, Sequence

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libmfa.so")

MFA_OK = 0
MFA_ERR_INVALID_ARG = 1
MFA_ERR_UNSUPPORTED = 2
MFA_ERR_WORKSPACE = 3
MFA_ERR_CUDA = 4
MFA_ERR_DEVICE_CHECK = 5

MFA_KV_BF16 = 0
MFA_KV_FP8_E4M3 = 1
MFA_KV_MXFP4 = 2
# the cache formats by the names the input generator uses
KV_DTYPES = {"bf16": MFA_KV_BF16, "fp8_e4m3": MFA_KV_FP8_E4M3, "mxfp4": MFA_KV_MXFP4}

MFA_OUT_BF16 = 0
MFA_OUT_FP32 = 1

MFA_DEV_TIMEOUT = 0x1
MFA_DEV_BAD_BLOCK = 0x2
MFA_DEV_BAD_LENGTH = 0x4
MFA_DEV_SCHEDULE = 0x8
MFA_DEV_RANGE = 0x10

MFA_PLAN_CHECK = 0x1
MFA_PLAN_NO_COMBINE = 0x2
MFA_PLAN_EARLY_METADATA = 0x4

NUM_Q_HEADS = 64
HEAD_DIM = 256
PAGE_SIZE = 64

# Every symbol include/mfa.h declares.
EXPORTED_SYMBOLS = ("mfa_decode_plan", "mfa_decode_run", "mfa_combine", "mfa_read_device_status",
                    "mfa_status_string", "mfa_abi_version", "mfa_last_cuda_error",
                    "mfa_decode_run_static_workspace", "mfa_kv_append", "mfa_decode_run_host",
                    "mfa_decode_append_run")

# Size of the library's own scratch array used by mfa_decode_run_static_workspace.
MFA_STATIC_WORKSPACE_BYTES = 24 * 1024 * 1024


class MfaProblem(ctypes.Structure):
    _fields_ = [("batch", ctypes.c_int32), ("num_q_heads", ctypes.c_int32),
                ("head_dim", ctypes.c_int32), ("page_size", ctypes.c_int32),
                ("max_pages_per_seq", ctypes.c_int32), ("num_blocks", ctypes.c_int32),
                ("kv_dtype", ctypes.c_int32), ("softmax_scale", ctypes.c_float),
                ("out_dtype", ctypes.c_int32), ("tokens_per_seq", ctypes.c_int32),
                ("num_kv_heads", ctypes.c_int32), ("kv_shared", ctypes.c_int32)]


class MfaPlan(ctypes.Structure):
    _fields_ = [("num_ctas", ctypes.c_int32), ("tile_tokens", ctypes.c_int32),
                ("max_tiles_per_cta", ctypes.c_int32), ("num_partials", ctypes.c_int32),
                ("batch", ctypes.c_int32), ("kv_dtype", ctypes.c_int32),
                ("flags", ctypes.c_uint32), ("num_sms", ctypes.c_int32),
                ("total_tiles", ctypes.c_uint64), ("workspace_bytes", ctypes.c_uint64),
                ("tokens_per_seq", ctypes.c_int32)]


class MfaError(RuntimeError):
    def __init__(self, status: int, where: str):
        msg = f"{where}: {status_string(status)} (status {status})"
        if status == MFA_ERR_CUDA and _lib is not None:
            msg += ": " + _lib.mfa_last_cuda_error().decode()
        super().__init__(msg)
        self.status = status


_lib = None


def load_library(path: str = LIB_PATH):
    """Load libmfa.so; raises if it has not been built (no fallback path exists)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise ImportError(f"{path} is missing: build it with decode_attention_02_gb300.build.build_library()")
    lib = ctypes.CDLL(path)
    P = ctypes.c_void_p
    lib.mfa_decode_plan.argtypes = [ctypes.POINTER(MfaProblem), P, ctypes.c_int32, ctypes.c_int32,
                                    ctypes.c_int32, ctypes.c_uint32, ctypes.POINTER(MfaPlan)]
    lib.mfa_decode_plan.restype = ctypes.c_int
    lib.mfa_decode_run.argtypes = [ctypes.POINTER(MfaPlan), ctypes.POINTER(MfaProblem), P, P, P, P, P, P, P,
                                   P, P, P, ctypes.c_uint64, P]
    lib.mfa_decode_run.restype = ctypes.c_int
    lib.mfa_combine.argtypes = [ctypes.POINTER(MfaPlan), ctypes.POINTER(MfaProblem), P, ctypes.c_uint64, P, P,
                                P, P]
    lib.mfa_combine.restype = ctypes.c_int
    lib.mfa_read_device_status.argtypes = [P, ctypes.POINTER(ctypes.c_uint32), ctypes.c_int32, P]
    lib.mfa_read_device_status.restype = ctypes.c_int
    lib.mfa_status_string.argtypes = [ctypes.c_int]
    lib.mfa_status_string.restype = ctypes.c_char_p
    lib.mfa_abi_version.argtypes = []
    lib.mfa_abi_version.restype = ctypes.c_int32
    lib.mfa_last_cuda_error.argtypes = []
    lib.mfa_last_cuda_error.restype = ctypes.c_char_p
    lib.mfa_decode_run_static_workspace.argtypes = [ctypes.POINTER(MfaPlan), ctypes.POINTER(MfaProblem), P, P, P,
                                                    P, P, P, P, P, P, P]
    lib.mfa_decode_run_static_workspace.restype = ctypes.c_int
    lib.mfa_kv_append.argtypes = [ctypes.POINTER(MfaProblem), P, P, P, P, P, P, P, P, P, P]
    lib.mfa_kv_append.restype = ctypes.c_int
    lib.mfa_decode_run_host.argtypes = [ctypes.POINTER(MfaPlan), ctypes.POINTER(MfaProblem), P, P, P, P, P,
                                        P, P, P, P, P, P, P, P, P, P, ctypes.c_uint64, P]
    lib.mfa_decode_run_host.restype = ctypes.c_int
    lib.mfa_decode_append_run.argtypes = [ctypes.POINTER(MfaPlan), ctypes.POINTER(MfaProblem), P, P, P, P, P, P, P,
                                          P, P, P, P, P, P, ctypes.c_uint64, P]
    lib.mfa_decode_append_run.restype = ctypes.c_int
    _lib = lib
    return lib


def status_string(status: int) -> str:
    try:
        return load_library().mfa_status_string(int(status)).decode()
    except ImportError:
        return "library not loaded"


def _check(status: int, where: str):
    if status != MFA_OK:
        raise MfaError(status, where)


def _ptr(x) -> Optional[int]:
    """Device pointer of a torch tensor (must be CUDA and contiguous), an int, or None."""
    if x is None:
        return None
    if isinstance(x, int):
        return x
    if not x.is_cuda:
        raise ValueError("expected a CUDA tensor")
    if not x.is_contiguous():
        raise ValueError("expected a contiguous tensor")
    return x.data_ptr()


def _nbytes(x) -> int:
    return x.numel() * x.element_size()


def _stream(stream) -> Optional[int]:
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


# The attention shapes the library runs: (num_q_heads, head_dim, num_kv_heads, kv_shared).
SHAPE_MFA = (64, 256, 1, False)     # Step-3's MFA: one shared K head and one shared V head
SHAPE_GQA = (64, 128, 4, False)     # grouped-query attention: 4 key/value heads of 128
SHAPE_MLA = (128, 512, 1, True)     # one 512-wide latent that is both key and value


def make_problem(batch: int, max_pages_per_seq: int, num_blocks: int, kv_dtype: int = MFA_KV_BF16,
                 softmax_scale: Optional[float] = None, num_q_heads: int = NUM_Q_HEADS,
                 head_dim: int = HEAD_DIM, page_size: int = PAGE_SIZE, out_dtype: int = MFA_OUT_BF16,
                 tokens_per_seq: int = 1, num_kv_heads: int = 1, kv_shared: bool = False) -> MfaProblem:
    if softmax_scale is None:
        softmax_scale = head_dim ** -0.5
    return MfaProblem(batch, num_q_heads, head_dim, page_size, max_pages_per_seq, num_blocks, kv_dtype,
                      softmax_scale, out_dtype, tokens_per_seq, num_kv_heads, 1 if kv_shared else 0)


def mfa_decode_plan(problem: MfaProblem, host_seq_lens: Optional[Sequence[int]] = None, max_seq_len: int = 0,
                    num_sms: int = 0, force_ctas: int = 0, flags: int = 0) -> MfaPlan:
    lib = load_library()
    plan = MfaPlan()
    lens_arr = None
    if host_seq_lens is not None:
        vals = [int(v) for v in host_seq_lens]
        lens_arr = (ctypes.c_int32 * max(1, len(vals)))(*vals)
    st = lib.mfa_decode_plan(ctypes.byref(problem), lens_arr, int(max_seq_len), int(num_sms), int(force_ctas),
                             int(flags), ctypes.byref(plan))
    _check(st, "mfa_decode_plan")
    return plan


def mfa_decode_run(plan: MfaPlan, problem: MfaProblem, q, k_cache, v_cache, k_scale, v_scale, block_table,
                   seq_lens, out, lse, workspace, stream=None, workspace_bytes: Optional[int] = None) -> None:
    lib = load_library()
    if workspace_bytes is None:
        workspace_bytes = _nbytes(workspace)
    st = lib.mfa_decode_run(ctypes.byref(plan), ctypes.byref(problem), _ptr(q), _ptr(k_cache), _ptr(v_cache),
                            _ptr(k_scale), _ptr(v_scale), _ptr(block_table), _ptr(seq_lens), _ptr(out),
                            _ptr(lse), _ptr(workspace), int(workspace_bytes), _stream(stream))
    _check(st, "mfa_decode_run")


def mfa_decode_append_run(plan: MfaPlan, problem: MfaProblem, q, k_cache, v_cache, k_scale, v_scale, block_table,
                          seq_lens, k_new, v_new, positions, out, lse, workspace, stream=None,
                          workspace_bytes: Optional[int] = None) -> None:
    """mfa_kv_append then mfa_decode_run in one call (one kernel for one new token per sequence)."""
    lib = load_library()
    if workspace_bytes is None:
        workspace_bytes = _nbytes(workspace)
    st = lib.mfa_decode_append_run(ctypes.byref(plan), ctypes.byref(problem), _ptr(q), _ptr(k_cache), _ptr(v_cache),
                                   _ptr(k_scale), _ptr(v_scale), _ptr(block_table), _ptr(seq_lens), _ptr(k_new),
                                   _ptr(v_new), _ptr(positions), _ptr(out), _ptr(lse), _ptr(workspace),
                                   int(workspace_bytes), _stream(stream))
    _check(st, "mfa_decode_append_run")


def mfa_decode_run_static_workspace(plan: MfaPlan, problem: MfaProblem, q, k_cache, v_cache, k_scale, v_scale,
                                    block_table, seq_lens, out, lse, stream=None) -> None:
    """mfa_decode_run with the library's own fixed scratch array instead of a workspace.

    For callers that must not allocate device memory; see include/mfa.h for the
    size limit and the rule that calls sharing a device must not overlap.
    """
    lib = load_library()
    st = lib.mfa_decode_run_static_workspace(ctypes.byref(plan), ctypes.byref(problem), _ptr(q), _ptr(k_cache),
                                             _ptr(v_cache), _ptr(k_scale), _ptr(v_scale), _ptr(block_table),
                                             _ptr(seq_lens), _ptr(out), _ptr(lse), _stream(stream))
    _check(st, "mfa_decode_run_static_workspace")


def _host_ptr(x) -> Optional[int]:
    """Address of a CPU torch tensor (contiguous), an int, or None."""
    if x is None:
        return None
    if isinstance(x, int):
        return x
    if x.is_cuda:
        raise ValueError("expected a CPU (pinned) tensor")
    if not x.is_contiguous():
        raise ValueError("expected a contiguous tensor")
    return x.data_ptr()


def mfa_decode_run_host(plan: MfaPlan, problem: MfaProblem, q_host, block_table_host, seq_lens_host, out_host,
                        lse_host, q_dev, block_table_dev, seq_lens_dev, out_dev, lse_dev, k_cache, v_cache, k_scale,
                        v_scale, workspace, stream=None, workspace_bytes: Optional[int] = None) -> None:
    """One decode step from host buffers (copies in, decode, copies out on one stream)."""
    lib = load_library()
    if workspace_bytes is None:
        workspace_bytes = _nbytes(workspace)
    st = lib.mfa_decode_run_host(ctypes.byref(plan), ctypes.byref(problem), _host_ptr(q_host),
                                 _host_ptr(block_table_host), _host_ptr(seq_lens_host), _host_ptr(out_host),
                                 _host_ptr(lse_host), _ptr(q_dev), _ptr(block_table_dev), _ptr(seq_lens_dev),
                                 _ptr(out_dev), _ptr(lse_dev), _ptr(k_cache), _ptr(v_cache), _ptr(k_scale),
                                 _ptr(v_scale), _ptr(workspace), int(workspace_bytes), _stream(stream))
    _check(st, "mfa_decode_run_host")


def mfa_combine(plan: MfaPlan, problem: MfaProblem, workspace, seq_lens, out, lse, stream=None,
                workspace_bytes: Optional[int] = None) -> None:
    lib = load_library()
    if workspace_bytes is None:
        workspace_bytes = _nbytes(workspace)
    st = lib.mfa_combine(ctypes.byref(plan), ctypes.byref(problem), _ptr(workspace), int(workspace_bytes),
                         _ptr(seq_lens), _ptr(out), _ptr(lse), _stream(stream))
    _check(st, "mfa_combine")


def mfa_kv_append(problem: MfaProblem, k_new, v_new, positions, block_table, k_cache, v_cache, k_scale=None,
                  v_scale=None, device_status=None, stream=None) -> None:
    """Write each sequence's new key/value row into the paged cache (FP8: quantised).

    k_new/v_new: bf16 [B*T, 256] (T = problem.tokens_per_seq new rows per sequence);
    positions: int32 [B] (index of each sequence's first new row, < 0 = none);
    device_status: a uint32 device tensor (or a decode workspace, whose first word is
    the status word) that collects bad-position / bad-page bits, or None.
    """
    lib = load_library()
    st = lib.mfa_kv_append(ctypes.byref(problem), _ptr(k_new), _ptr(v_new), _ptr(positions), _ptr(block_table),
                           _ptr(k_cache), _ptr(v_cache), _ptr(k_scale), _ptr(v_scale), _ptr(device_status),
                           _stream(stream))
    _check(st, "mfa_kv_append")


def mfa_read_device_status(workspace, clear: bool = True, stream=None) -> int:
    lib = load_library()
    word = ctypes.c_uint32(0)
    st = lib.mfa_read_device_status(_ptr(workspace), ctypes.byref(word), 1 if clear else 0, _stream(stream))
    _check(st, "mfa_read_device_status")
    return int(word.value)


def workspace_layout(plan: MfaPlan, head_dim: int = HEAD_DIM):
    """Byte offsets of (partial O, partial lse) inside the workspace (see include/mfa.h)."""
    o_off = 256
    lse_off = (o_off + plan.num_partials * NUM_Q_HEADS * head_dim * 4 + 255) // 256 * 256
    return o_off, lse_off


class Decoder:
    """Plan + workspace for one batch shape; ``__call__`` enqueues a decode step.

    Device buffers come from PyTorch's allocator; the step itself is
    ``mfa_decode_run`` (decode kernel + combine kernel).
    """

    def __init__(self, batch: int, max_pages_per_seq: int, num_blocks: int, kv_dtype: int = MFA_KV_BF16,
                 softmax_scale: Optional[float] = None, host_seq_lens=None, max_seq_len: int = 0,
                 force_ctas: int = 0, flags: int = 0, device=None, out_dtype: int = MFA_OUT_BF16,
                 tokens_per_seq: int = 1, shape=SHAPE_MFA):
        import torch
        H, d, G, shared = shape
        self.problem = make_problem(batch, max_pages_per_seq, num_blocks, kv_dtype, softmax_scale,
                                    num_q_heads=H, head_dim=d, out_dtype=out_dtype, tokens_per_seq=tokens_per_seq,
                                    num_kv_heads=G, kv_shared=shared)
        if host_seq_lens is None and max_seq_len == 0:
            max_seq_len = max_pages_per_seq * PAGE_SIZE
        self.plan = mfa_decode_plan(self.problem, host_seq_lens, max_seq_len, 0, force_ctas, flags)
        self.device = torch.device("cuda") if device is None else torch.device(device)
        self.workspace = torch.zeros(int(self.plan.workspace_bytes), dtype=torch.uint8, device=self.device)

    def __call__(self, q, k_cache, v_cache, block_table, seq_lens, k_scale=None, v_scale=None, out=None,
                 lse=None, stream=None):
        import torch
        pr = self.problem
        rows = pr.batch * pr.tokens_per_seq   # (sequence, new token) pairs
        if out is None:
            dt = torch.float32 if pr.out_dtype == MFA_OUT_FP32 else torch.bfloat16
            out = torch.empty((rows, pr.num_q_heads, pr.head_dim), dtype=dt, device=q.device)
        if lse is None:
            lse = torch.empty((rows, pr.num_q_heads), dtype=torch.float32, device=q.device)
        mfa_decode_run(self.plan, self.problem, q, k_cache, v_cache, k_scale, v_scale, block_table, seq_lens,
                       out, lse, self.workspace, stream)
        return out, lse

    def run_host(self, q_host, block_table_host, seq_lens_host, out_host, lse_host, k_cache, v_cache, k_scale=None,
                 v_scale=None, stream=None):
        """One step from pinned host buffers into pinned host outputs (mfa_decode_run_host),
        on device staging buffers this decoder owns.  Asynchronous on ``stream``."""
        import torch
        if not hasattr(self, "_staging"):
            dev = self.device
            pr = self.problem
            B = pr.batch
            rows = B * pr.tokens_per_seq
            odt = torch.float32 if pr.out_dtype == MFA_OUT_FP32 else torch.bfloat16
            self._staging = dict(
                q=torch.empty((rows, pr.num_q_heads, pr.head_dim), dtype=torch.bfloat16, device=dev),
                table=torch.empty((B, pr.max_pages_per_seq), dtype=torch.int32, device=dev),
                lens=torch.empty((B,), dtype=torch.int32, device=dev),
                out=torch.empty((rows, pr.num_q_heads, pr.head_dim), dtype=odt, device=dev),
                lse=torch.empty((rows, pr.num_q_heads), dtype=torch.float32, device=dev))
        st = self._staging
        mfa_decode_run_host(self.plan, self.problem, q_host, block_table_host, seq_lens_host, out_host, lse_host,
                            st["q"], st["table"], st["lens"], st["out"], None if lse_host is None else st["lse"],
                            k_cache, v_cache, k_scale, v_scale, self.workspace, stream)
