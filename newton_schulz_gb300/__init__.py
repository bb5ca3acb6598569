"""GB300-native Muon optimizer step (momentum -> Newton-Schulz -> update).

The compute path is libmuon.so (hand-written sm_103a CUDA behind a C ABI,
declared in include/muon.h); ``binding`` marshals torch tensors into it.
Importing this package does not load the library; the first call does, and
fails loudly when it is missing.
"""
from .binding import (MuonError, muon_last_launch_count, muon_ns_batched,  # noqa: F401
                      muon_ns_batched_ex, muon_profile_enable, muon_profile_read,
                      muon_query_status, muon_release_workspace, muon_status_string,
                      muon_step_grouped, muon_step_grouped_ex)
