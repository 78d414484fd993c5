// Cost-model constants of pkv_policy_default. Written by serving_paged_gqa_gb300/calibrate.py (fit) from
// the calibration sweep; rebuild the library after changing them.
#pragma once
#define PKV_FIT_SOURCE "least squares on 2787 timed candidate plans, then regret-refined on every candidate, seeds [0, 1, 2, 3, 4]"
#define PKV_FIT_LAUNCH_US 6.68741
#define PKV_FIT_HBM_GBS 6800
#define PKV_FIT_CTA_GBS 27.9217
#define PKV_FIT_WQ_CTA_GBS 21.1042
#define PKV_FIT_TASK_US 0.298825
#define PKV_FIT_TAIL 1.21564
#define PKV_FIT_MERGE_US 3.03071
#define PKV_FIT_MERGE_STATE_US 0.0292293
#define PKV_FIT_FUSED_US 3.33189
#define PKV_FIT_FUSED_STATE_US 0.0375297
#define PKV_FIT_BUILD_US 4
