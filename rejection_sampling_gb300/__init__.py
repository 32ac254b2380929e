"""GB300-native batched lossless speculative verification.

The verification step of drafter-and-verifier decoding (Leviathan-style
rejection sampling) behind a C ABI (include/spec_verify.h) implemented by
hand-written CUDA kernels for sm_103a in libspec_verify.so:

  spec_verify_dense     dense logits: a streaming statistics kernel and a
                        cluster-per-row decision kernel (small vocabularies:
                        one warp per row)
  spec_verify_sparse    Uno-style sorted top-k (id, prob) support lists
  spec_verify_anyorder  masked-diffusion any-order window, small vocabulary
  spec_verify_greedy    greedy (temperature 0) verification: argmax match
  spec_commit_confident confidence-threshold commit of a block-diffusion pass
  spec_support_topk     sparse support lists (temperature, top-k, top-p)
  spec_verify_anyorder_rounds  windowed multi-round any-order verification
                        (several rounds on one window of draft distributions)
  spec_anyorder_window  the cosine-schedule window W(i) (host function)
  spec_verify_dense_static  spec_verify_dense on a static scratch array, for
                        callers that cannot allocate device memory

The Python functions below have the same names as the C entry points and only
marshal torch tensors; the library is loaded lazily on first use and every
call fails loudly if it is missing.  ``workloads`` generates the seeded
synthetic inputs.
"""
from ._binding import (  # noqa: F401
    EXPORTED, CommitResult, SupportResult, SV_BF16, SV_ERR_CUDA, SV_ERR_DEVICE_INPUT, SV_ERR_INVALID_ARG, SV_ERR_SCRATCH_LIMIT,
    SV_ERR_TIMEOUT, SV_ERR_UNSUPPORTED, SV_F32, SV_OK, SV_STATIC_SCRATCH_BYTES, SpecVerifyError,
    VerifyResult, abi_version, check,
    get_workspace, library_path, load, prepare_anyorder, prepare_commit, prepare_dense,
    prepare_greedy, prepare_support, spec_commit_confident, spec_support_topk,
    RoundsResult, prepare_rounds, spec_anyorder_window, spec_verify_anyorder_rounds,
    prepare_sparse, PreparedCall, spec_verify_anyorder, spec_verify_dense,
    spec_verify_dense_static, spec_verify_greedy, spec_verify_sparse, status_string,
    workspace_size,
)
from ._build import build  # noqa: F401
