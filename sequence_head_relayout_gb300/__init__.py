"""GB300-native exact destination-major relayouts around sequence-head attention."""
